// bwd_sm103.cu -- exact attention backward on sm_103a tensor cores.
//
// The backward recomputes the probabilities tile by tile from the saved
// log-sum-exp instead of storing S or P ("从Online-Softmax到FlashAttention
// V1/V2/V3" 0x04 and "LLM 注意力与计算内核精读笔记 · 02 FlashAttention" §6).
// Following FlashAttention-2's backward order (0x05 of the first page), K/V
// tiles are the outer loop (one CTA each) and query tiles the inner loop, so
// dK and dV stay on chip and only dQ is accumulated across CTAs.  The
// gradient of O = softmax(scale Q K^T) V given dO is, per (i, j):
//   p_ij = exp(s_ij - LSE_i),  dP_ij = <dO_i, v_j>,  dS_ij = p_ij (dP_ij - D_i),
//   dV_j += p_ij dO_i,  dK_j += scale dS_ij q_i,  dQ_i += scale dS_ij k_j,
// with D_i = <dO_i, O_i>.
//
// Kernels:
//   bwd_pre     D_i = rowsum(dO * O) and LSE_i * log2(e) into the workspace;
//               zeroes the fp32 dQ accumulator.
//   bwd_main    one CTA per (batch, kv head, 128-key tile); loops over the G
//               query heads of the group and the 64-row query tiles.  All
//               five products run on tcgen05 with TMEM accumulators:
//                 S^T  = K Q^T         (M=128 keys, N=64 queries)
//                 dP^T = V dO^T
//                 dV  += P^T dO        (P^T from TMEM, bf16)
//                 dK  += dS^T Q        (dS^T from TMEM, bf16)
//                 dQ^T = K^T dS^T      (dS^T from shared memory; M = d)
//               dK and dV stay in TMEM across the whole group (no atomics);
//               dQ^T is read back by a second warpgroup and reduce-added
//               (fp32) into the accumulator.
//   bwd_dq      dQ = bf16(scale * accumulator).
// Warps of bwd_main: 0 TMA producer, 1 TMEM allocator + MMA issuer,
// 2..5 probability/gradient math (thread = key row), 6..9 dQ readback
// (thread = head-dim index).
#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBK = 128;  // keys per CTA
constexpr int kBQ = 64;   // query rows per inner tile
constexpr int kMainThreads = 320;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Bwd {
  static constexpr int CB = D / 64;
  static constexpr int KBLK = kBK * 128;  // 128 rows x 128 bytes
  static constexpr int QBLK = kBQ * 128;  // 64 rows x 128 bytes
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + CB * KBLK;
  static constexpr int OFF_DS = OFF_V + CB * KBLK;  // dS^T, 128 keys x 64 queries bf16
  static constexpr int OFF_STAGE = OFF_DS + kBK * 128;
  static constexpr int ST_Q = 0;
  static constexpr int ST_DO = CB * QBLK;
  static constexpr int ST_LSE = 2 * CB * QBLK;
  static constexpr int ST_D = ST_LSE + kBQ * 4;
  static constexpr int STAGE_BYTES = (ST_D + kBQ * 4 + 1023) / 1024 * 1024;
  static constexpr int STAGES = 2;
  static constexpr int OFF_BAR = OFF_STAGE + STAGES * STAGE_BYTES;
  static constexpr int B_KVFULL = 0;
  static constexpr int B_STFULL = 1;               // STAGES
  static constexpr int B_STEMPTY = B_STFULL + STAGES;
  static constexpr int B_SFULL = B_STEMPTY + STAGES;
  static constexpr int B_DPFULL = B_SFULL + 1;
  static constexpr int B_PFULL = B_DPFULL + 1;
  static constexpr int B_DSFULL = B_PFULL + 1;
  static constexpr int B_DQFULL = B_DSFULL + 1;
  static constexpr int B_DQFREE = B_DQFULL + 1;
  static constexpr int B_MMADONE = B_DQFREE + 1;
  static constexpr int B_DRAIN = B_MMADONE + 1;
  static constexpr int NBARS = B_DRAIN + 1;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;
  // TMEM columns
  static constexpr uint32_t TM_DV = 0;
  static constexpr uint32_t TM_DK = D;
  static constexpr uint32_t TM_S = 2 * D;
  static constexpr uint32_t TM_DP = 2 * D + 64;
  static constexpr uint32_t TM_DQ = 2 * D + 128;
  static constexpr uint32_t IDESC_ST = idesc_bf16(128, kBQ, false, false);
  static constexpr uint32_t IDESC_KV = idesc_bf16(128, D, false, true);
  static constexpr uint32_t IDESC_DQ = idesc_bf16(128, kBQ, true, true);
};

// ------------------------------------------------------------------ preprocess
// One warp per (b, h, row) of the padded row range: D, LSE2, and a zeroed
// accumulator row.  Rows past N get D = 0 and LSE2 = +inf (probability 0).
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdParams p) {
  constexpr int EPL = D / 32;  // elements per lane
  const long long rows = (long long)p.B * p.Hq * p.Npad;
  const int lane = threadIdx.x & 31;
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
       r += ((long long)gridDim.x * blockDim.x) >> 5) {
    const long long bh = r / p.Npad;
    const int i = (int)(r - bh * p.Npad);
    float dsum = 0.f;
    if (i < p.N) {
      const size_t off = ((size_t)bh * p.N + i) * D + lane * EPL;
      if (EPL == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(p.O + off);
        const uint2 g = *reinterpret_cast<const uint2*>(p.dO + off);
        const uint32_t aw[2] = {a.x, a.y}, gw[2] = {g.x, g.y};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          dsum += __uint_as_float(aw[k] << 16) * __uint_as_float(gw[k] << 16);
          dsum += __uint_as_float(aw[k] & 0xffff0000u) * __uint_as_float(gw[k] & 0xffff0000u);
        }
      } else {
        const uint32_t a = *reinterpret_cast<const uint32_t*>(p.O + off);
        const uint32_t g = *reinterpret_cast<const uint32_t*>(p.dO + off);
        dsum += __uint_as_float(a << 16) * __uint_as_float(g << 16);
        dsum += __uint_as_float(a & 0xffff0000u) * __uint_as_float(g & 0xffff0000u);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
    if (lane == 0) {
      p.Dvec[r] = dsum;
      p.LSE2[r] = i < p.N ? p.LSE[bh * p.N + i] * 1.4426950408889634f : INFINITY;
    }
    float4* acc = reinterpret_cast<float4*>(p.dQacc + r * D);
    for (int k = lane; k < D / 4; k += 32) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ------------------------------------------------------------------ dQ convert
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const BwdParams p) {
  const long long total = (long long)p.B * p.Hq * p.N * (D / 4);
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total;
       v += (long long)gridDim.x * blockDim.x) {
    const long long e = v * 4;
    const long long row = e / D;  // (b*Hq + h) * N + i
    const int col = (int)(e - row * D);
    const long long bh = row / p.N;
    const long long i = row - bh * p.N;
    const float4 a = *reinterpret_cast<const float4*>(p.dQacc + (bh * p.Npad + i) * D + col);
    uint2 o;
    o.x = pack_bf16(a.x * p.scale, a.y * p.scale);
    o.y = pack_bf16(a.z * p.scale, a.w * p.scale);
    *reinterpret_cast<uint2*>(p.dQ + row * D + col) = o;
  }
}

// ------------------------------------------------------------------ main
template <int D>
__global__ void __launch_bounds__(kMainThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const BwdParams p) {
  using C = Bwd<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V, sDS = sb + C::OFF_DS;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA -> (b * Hkv + hk, key tile): the key tiles of a few kv heads run together
  // so that their query-side operands and dQ accumulator stay in L2; within a
  // group, key tile 0 (the most query tiles when causal) comes first.
  int bhk, jt;
  grouped_order(blockIdx.x, p.B * p.Hkv, (p.N + kBK - 1) / kBK, p.head_group, bhk, jt);
  const int k0 = jt * kBK;
  const int b = bhk / p.Hkv;
  const int hk = bhk - b * p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int n_q = (p.N + kBQ - 1) / kBQ;
  const int i0 = p.causal ? min(n_q, (k0 / kBQ)) : 0;  // first query tile that sees these keys
  const int per_head = n_q - i0;
  const int T = G * per_head;  // inner iterations

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KVFULL), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::B_STFULL + s), 1);
      mbar_init(bar(C::B_STEMPTY + s), 1);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_PFULL), 128);
    mbar_init(bar(C::B_DSFULL), 128);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQFREE), 128);
    mbar_init(bar(C::B_MMADONE), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.wait_limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::CB * C::KBLK);
      for (int cb = 0; cb < C::CB; ++cb) {
        tma_load_3d(sK + cb * C::KBLK, &tmK, bar(C::B_KVFULL), cb * 64, k0, bhk);
        tma_load_3d(sV + cb * C::KBLK, &tmV, bar(C::B_KVFULL), cb * 64, k0, bhk);
      }
      int t = 0;
      for (; t < T; ++t) {
        const int s = t % C::STAGES;
        if (t >= C::STAGES && !mbar_wait(bar(C::B_STEMPTY + s), ((t / C::STAGES) & 1) ^ 1, wc)) break;
        const int g = t / per_head;
        const int it = i0 + (t - g * per_head);
        const int bhq = b * p.Hq + hk * G + g;
        const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE_BYTES;
        const uint32_t fb = bar(C::B_STFULL + s);
        mbar_arrive_expect_tx(fb, 2 * C::CB * C::QBLK + 2 * kBQ * 4);
        for (int cb = 0; cb < C::CB; ++cb) {
          tma_load_3d(st + C::ST_Q + cb * C::QBLK, &tmQ, fb, cb * 64, it * kBQ, bhq);
          tma_load_3d(st + C::ST_DO + cb * C::QBLK, &tmdO, fb, cb * 64, it * kBQ, bhq);
        }
        const size_t vo = (size_t)bhq * p.Npad + (size_t)it * kBQ;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                st + C::ST_LSE),
            "l"(p.LSE2 + vo), "r"(kBQ * 4), "r"(fb)
            : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                st + C::ST_D),
            "l"(p.Dvec + vo), "r"(kBQ * 4), "r"(fb)
            : "memory");
      }
      mbar_wait_drain(bar(C::B_KVFULL), 0, wc);
      for (int k = max(0, t - C::STAGES); k < t; ++k)
        mbar_wait_drain(bar(C::B_STFULL + k % C::STAGES), (k / C::STAGES) & 1, wc);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    {
      // The whole warp runs this loop (uniform operands); one elected lane issues.
      bool ok = mbar_wait_warp(bar(C::B_KVFULL), 0, wc);
      for (int t = 0; t < T && ok; ++t) {
        const int s = t % C::STAGES;
        const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE_BYTES;
        if (!mbar_wait_warp(bar(C::B_STFULL + s), (t / C::STAGES) & 1, wc)) break;
        // All MMAs of the previous iteration are complete: the S/P, dP/dS
        // TMEM regions and the dS shared-memory tile may be overwritten.
        if (t > 0 && !mbar_wait_warp(bar(C::B_MMADONE), (t - 1) & 1, wc)) break;
        tc_fence_after();
        // S^T = K Q^T and dP^T = V dO^T (both K-major operands).
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * C::KBLK + (kk & 3) * 32;
          const uint32_t qa = (kk >> 2) * C::QBLK + (kk & 3) * 32;
          mma_ss_warp(tmem + C::TM_S, sdesc_sw128(sK + ka, 16, 1024), sdesc_sw128(st + C::ST_Q + qa, 16, 1024),
                 C::IDESC_ST, kk > 0);
        }
        tc_commit_warp(bar(C::B_SFULL));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * C::KBLK + (kk & 3) * 32;
          const uint32_t qa = (kk >> 2) * C::QBLK + (kk & 3) * 32;
          mma_ss_warp(tmem + C::TM_DP, sdesc_sw128(sV + ka, 16, 1024),
                 sdesc_sw128(st + C::ST_DO + qa, 16, 1024), C::IDESC_ST, kk > 0);
        }
        tc_commit_warp(bar(C::B_DPFULL));
        // dV += P^T dO  (A = P^T in TMEM, B = dO MN-major: 16 query rows = 2048 bytes)
        if (!mbar_wait_warp(bar(C::B_PFULL), t & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_ts_warp(tmem + C::TM_DV, tmem + C::TM_S + kk * 8,
                 sdesc_sw128(st + C::ST_DO + kk * 2048, C::QBLK, 1024), C::IDESC_KV,
                 (t > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q
        if (!mbar_wait_warp(bar(C::B_DSFULL), t & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_ts_warp(tmem + C::TM_DK, tmem + C::TM_DP + kk * 8,
                 sdesc_sw128(st + C::ST_Q + kk * 2048, C::QBLK, 1024), C::IDESC_KV,
                 (t > 0 || kk > 0) ? 1u : 0u);
        // dQ^T = K^T dS^T  (A = K as MN-major [d x keys], B = dS^T MN-major [keys x queries]).
        // For d = 64 the instruction still has M = 128; lanes 64..127 read the
        // V tile as filler and are ignored.
        if (t > 0 && !mbar_wait_warp(bar(C::B_DQFREE), (t - 1) & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_ss_warp(tmem + C::TM_DQ, sdesc_sw128(sK + kk * 2048, C::KBLK, 1024),
                 sdesc_sw128(sDS + kk * 2048, 8192, 1024), C::IDESC_DQ, kk > 0);
        tc_commit_warp(bar(C::B_DQFULL));
        tc_commit_warp(bar(C::B_STEMPTY + s));
        tc_commit_warp(bar(C::B_MMADONE));
      }
      tc_commit_warp(bar(C::B_DRAIN));
      mbar_wait_drain_warp(bar(C::B_DRAIN), 0, wc);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ P / dS math
    const int quad = warp & 3;
    const int kr = quad * 32 + lane;  // key row within the tile
    const int key = k0 + kr;
    const bool key_ok = key < p.N;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t % C::STAGES;
      const int g = t / per_head;
      const int it = i0 + (t - g * per_head);
      const int q0 = it * kBQ;
      const uint32_t stp = sb + C::OFF_STAGE + s * C::STAGE_BYTES;
      if (!mbar_wait(bar(C::B_STFULL + s), (t / C::STAGES) & 1, wc) ||
          !mbar_wait(bar(C::B_SFULL), t & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(tmem + lane_off + C::TM_S, sr[0]);
      tmem_ld32(tmem + lane_off + C::TM_S + 32, sr[1]);
      tmem_ld_wait(sr[0]);
      reg_fence32(sr[1]);
      const bool diag = p.causal && (q0 < k0 + kBK - 1);
      float pv[64];
      uint32_t pk[32];
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 lq = lds_f4(stp + C::ST_LSE + 16 * c4);  // same address in every lane
        const float l4[4] = {lq.x, lq.y, lq.z, lq.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = 4 * c4 + u;
          float x = ex2(fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, -l4[u]));
          if (!key_ok || (diag && key > q0 + c)) x = 0.f;
          pv[c] = x;
        }
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) pk[c] = pack_bf16(pv[2 * c], pv[2 * c + 1]);
      tmem_st32(tmem + lane_off + C::TM_S, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_PFULL));

      if (!mbar_wait(bar(C::B_DPFULL), t & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dS = P (dP - D), one half of the 64 query columns at a time.
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t dr[32];
        tmem_ld32(tmem + lane_off + C::TM_DP + 32 * half, dr);
        tmem_ld_wait(dr);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 dq = lds_f4(stp + C::ST_D + 128 * half + 16 * c4);
          const int c = 32 * half + 4 * c4;
          pk[16 * half + 2 * c4] = pack_bf16(pv[c] * (__uint_as_float(dr[4 * c4]) - dq.x),
                                             pv[c + 1] * (__uint_as_float(dr[4 * c4 + 1]) - dq.y));
          pk[16 * half + 2 * c4 + 1] = pack_bf16(pv[c + 2] * (__uint_as_float(dr[4 * c4 + 2]) - dq.z),
                                                 pv[c + 3] * (__uint_as_float(dr[4 * c4 + 3]) - dq.w));
        }
      }
      tmem_st32(tmem + lane_off + C::TM_DP, pk);
      // dS^T row into shared memory for the dQ product (128-byte swizzle: the
      // 16-byte chunk c of row kr lives at chunk position c ^ (kr & 7)).
      if (t > 0 && !mbar_wait(bar(C::B_DQFULL), (t - 1) & 1, wc)) {
        ok = false;
        break;
      }
      const uint32_t dsrow = sDS + kr * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        sts_u4(dsrow + ((c ^ (kr & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_DSFULL));
    }
    // Epilogue: dV and scale * dK rows of this key tile.
    if (ok && T > 0 && mbar_wait(bar(C::B_MMADONE), (T - 1) & 1, wc)) {
      tc_fence_after();
      const size_t row = (size_t)bhk * p.N + key;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        uint16_t* dst = (which == 0 ? p.dV : p.dK) + row * D;
        const float mul = which == 0 ? 1.f : p.scale;
        const uint32_t base = which == 0 ? C::TM_DV : C::TM_DK;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + base + c * 32, o);
          tmem_ld_wait(o);
          if (key_ok) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(o[8 * i + 0]) * mul, __uint_as_float(o[8 * i + 1]) * mul);
              v.y = pack_bf16(__uint_as_float(o[8 * i + 2]) * mul, __uint_as_float(o[8 * i + 3]) * mul);
              v.z = pack_bf16(__uint_as_float(o[8 * i + 4]) * mul, __uint_as_float(o[8 * i + 5]) * mul);
              v.w = pack_bf16(__uint_as_float(o[8 * i + 6]) * mul, __uint_as_float(o[8 * i + 7]) * mul);
              d4[i] = v;
            }
          }
        }
      }
    } else if (T == 0 && key_ok) {
      // No query tile reaches these keys (cannot happen when Nq = Nk): zero grads.
      const size_t row = (size_t)bhk * p.N + key;
      for (int c = 0; c < D; ++c) p.dV[row * D + c] = p.dK[row * D + c] = 0;
    }
  } else {
    // ------------------------------------------------------------ dQ readback
    const int quad = warp & 3;
    const int dcol = quad * 32 + lane;  // head-dim index (TMEM lane of dQ^T)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    for (int t = 0; t < T; ++t) {
      const int g = t / per_head;
      const int it = i0 + (t - g * per_head);
      const int bhq = b * p.Hq + hk * G + g;
      if (!mbar_wait(bar(C::B_DQFULL), t & 1, wc)) break;
      tc_fence_after();
      uint32_t r[2][32];
      tmem_ld32(tmem + lane_off + C::TM_DQ, r[0]);
      tmem_ld32(tmem + lane_off + C::TM_DQ + 32, r[1]);
      tmem_ld_wait(r[0]);
      reg_fence32(r[1]);
      tc_fence_before();
      mbar_arrive(bar(C::B_DQFREE));
      if (dcol < D) {
        float* acc = p.dQacc + ((size_t)bhq * p.Npad + (size_t)it * kBQ) * D + dcol;
#pragma unroll
        for (int c = 0; c < kBQ; ++c) atomicAdd(acc + (size_t)c * D, __uint_as_float(r[c >> 5][c & 31]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                   const CUtensorMap& tmdO, const BwdParams& p, unsigned stages,
                   cudaStream_t stream) {
  using C = Bwd<D>;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = cudaSuccess;
  if (stages & kBwdPre) {
    const long long rows = (long long)p.B * p.Hq * p.Npad;
    const int pre_blocks = (int)std::min<long long>((rows + 7) / 8, (long long)sms * 16);
    bwd_pre_kernel<D><<<pre_blocks, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (stages & kBwdMain) {
    auto kern = bwd_main_kernel<D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(p.B * p.Hkv * ((p.N + kBK - 1) / kBK));
    kern<<<grid, kMainThreads, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, tmdO, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (stages & kBwdConvert) {
    const long long vec = (long long)p.B * p.Hq * p.N * (D / 4);
    const int cv_blocks = (int)std::min<long long>((vec + 255) / 256, (long long)sms * 16);
    bwd_dq_kernel<D><<<cv_blocks, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return e;
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int N, int d) {
  const size_t Npad = (size_t)(N + 63) / 64 * 64;
  const size_t rows = (size_t)B * Hq * Npad;
  return (rows * d * 4 + 255) / 256 * 256 + 2 * ((rows * 4 + 255) / 256 * 256);
}

cudaError_t launch_bwd_bf16(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO, const BwdParams& p,
                            unsigned stages, cudaStream_t stream) {
  if (d == 128) return launch<128>(tmQ, tmK, tmV, tmdO, p, stages, stream);
  if (d == 64) return launch<64>(tmQ, tmK, tmV, tmdO, p, stages, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
