// fwd_sm103.cu -- exact attention forward on sm_103a tensor cores.
//
// Computes O = softmax(scale * Q K^T [+ causal mask]) V and LSE per query row
// with the online (m, l, O) merge of "LLM 注意力与计算内核精读笔记 · 02
// FlashAttention" §5: per K/V tile, m+ = max(m, m~), l+ = e^{m-m+} l + rowsum(P~),
// O+ = e^{m-m+} O + P~ V.  As in FlashAttention-2 ("从Online-Softmax到
// FlashAttention V1/V2/V3", 0x05), O stays unnormalised and 1/l is applied
// once at the end; each CTA owns one 128-row query tile and loops over K/V
// (Q outer loop), so CTAs never communicate.  Causal tiles above the diagonal
// are never visited and only the diagonal tile is masked (0x09's three tile
// cases).  GQA reads K/V head h / (Hq / Hkv) by indexing (0x09).
//
// Mapping to the hardware (one CTA, 6 warps):
//   warp 0      TMA producer: Q tile once, then K_j, V_j through a STAGES-deep
//               ring of shared-memory slots (mbarrier full/empty pairs).
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//               S_j = Q K_j^T  (SS MMA, M=128 N=128, into TMEM buffer j%2)
//               O  += P_j V_j  (TS MMA, P read from TMEM, V from shared memory)
//   warps 2..5  softmax: thread r owns query row r; it reads its S row from
//               TMEM (32x32b loads), keeps m and l in registers in log2 units,
//               writes P as packed bf16 over the first 64 columns of the same
//               S buffer, rescales its O row in TMEM when the max moved, and
//               finally writes O / l and LSE.
// TMEM columns: [0,128) S/P buffer 0, [128,256) buffer 1, [256,256+d) O.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;  // query rows per CTA
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Fwd {
  static constexpr int CB = D / 64;              // 128-byte column blocks per row
  static constexpr int BLOCK_BYTES = 128 * 128;  // one 128-row x 64-col bf16 block
  static constexpr int TILE_BYTES = CB * BLOCK_BYTES;
  static constexpr int STAGES = D == 128 ? 4 : 6;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = TILE_BYTES;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TILE_BYTES;
  // barrier indices
  static constexpr int B_QFULL = 0;
  static constexpr int B_KVFULL = 1;
  static constexpr int B_KVEMPTY = B_KVFULL + STAGES;
  static constexpr int B_SFULL = B_KVEMPTY + STAGES;  // 2
  static constexpr int B_PFULL = B_SFULL + 2;         // 2
  static constexpr int B_ODONE = B_PFULL + 2;
  static constexpr int B_DRAIN = B_ODONE + 1;
  static constexpr int NBARS = B_DRAIN + 1;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;  // + alignment slack
  static constexpr uint32_t IDESC_S = idesc_bf16(kBM, kBN, false, false);
  static constexpr uint32_t IDESC_O = idesc_bf16(kBM, D, false, true);
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 256;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Fwd<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q;
  const uint32_t sKV = sb + C::OFF_KV;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;                      // b * Hq + h
  const int tile = p.n_qtiles - 1 - (int)blockIdx.y;  // heaviest causal tiles launch first
  const int q0 = tile * kBM;
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int bh_kv = b * p.Hkv + h / (p.Hq / p.Hkv);
  int n_kv = (p.N + kBN - 1) / kBN;
  if (p.causal) n_kv = min(n_kv, tile + 1);  // tiles right of the diagonal are skipped

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QFULL), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::B_KVFULL + s), 1);
      mbar_init(bar(C::B_KVEMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_SFULL + i), 1);
      mbar_init(bar(C::B_PFULL + i), kBM);
    }
    mbar_init(bar(C::B_ODONE), 1);
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
      mbar_arrive_expect_tx(bar(C::B_QFULL), C::TILE_BYTES);
      for (int cb = 0; cb < C::CB; ++cb)
        tma_load_3d(sQ + cb * C::BLOCK_BYTES, &tmQ, bar(C::B_QFULL), cb * 64, q0, bh);
      int li = 0;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        for (int t = 0; t < 2; ++t, ++li) {
          const int s = li % C::STAGES;
          const uint32_t ph = (li / C::STAGES) & 1;
          if (li >= C::STAGES && !mbar_wait(bar(C::B_KVEMPTY + s), ph ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::B_KVFULL + s), C::TILE_BYTES);
          const CUtensorMap* m = t ? &tmV : &tmK;
          for (int cb = 0; cb < C::CB; ++cb)
            tma_load_3d(sKV + s * C::TILE_BYTES + cb * C::BLOCK_BYTES, m, bar(C::B_KVFULL + s),
                        cb * 64, j * kBN, bh_kv);
        }
      }
      // Drain: every issued copy must land before the CTA may exit.
      mbar_wait_drain(bar(C::B_QFULL), 0, wc);
      for (int k = max(0, li - C::STAGES); k < li; ++k)
        mbar_wait_drain(bar(C::B_KVFULL + k % C::STAGES), (k / C::STAGES) & 1, wc);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(bar(C::B_QFULL), 0, wc);
      tc_fence_after();
      auto issue_s = [&](int jj) -> bool {
        const int li = 2 * jj;
        const int s = li % C::STAGES;
        if (!mbar_wait(bar(C::B_KVFULL + s), (li / C::STAGES) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t d_t = tmem + C::TM_S + (jj & 1) * 128;
        const uint32_t kb = sKV + s * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32;
          mma_ss(d_t, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), C::IDESC_S,
                 kk > 0);
        }
        tc_commit(bar(C::B_SFULL + (jj & 1)));
        tc_commit(bar(C::B_KVEMPTY + s));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int jj = 0; jj < n_kv && ok; ++jj) {
        if (jj + 1 < n_kv) {
          // S buffer (jj+1)&1 held P_{jj-1}; PV_{jj-1} must have consumed it.
          if (jj >= 1 && !mbar_wait(bar(C::B_ODONE), (jj - 1) & 1, wc)) break;
          if (!issue_s(jj + 1)) break;
        }
        if (!mbar_wait(bar(C::B_PFULL + (jj & 1)), (jj >> 1) & 1, wc)) break;
        tc_fence_after();
        const int li = 2 * jj + 1;
        const int s = li % C::STAGES;
        if (!mbar_wait(bar(C::B_KVFULL + s), (li / C::STAGES) & 1, wc)) break;
        tc_fence_after();
        const uint32_t vb = sKV + s * C::TILE_BYTES;
        const uint32_t p_t = tmem + C::TM_S + (jj & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // A: 16 keys of P = 8 TMEM columns of packed bf16 pairs.
          // B: V rows 16kk..16kk+15, MN-major (d contiguous), 2048 bytes per 16 rows.
          mma_ts(tmem + C::TM_O, p_t + kk * 8, sdesc_sw128(vb + kk * 2048, C::BLOCK_BYTES, 1024),
                 C::IDESC_O, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(C::B_ODONE));
        tc_commit(bar(C::B_KVEMPTY + s));
      }
      // Drain: all MMAs of this thread complete before TMEM is released.
      tc_commit(bar(C::B_DRAIN));
      mbar_wait_drain(bar(C::B_DRAIN), 0, wc);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quad * 32 + lane;
    const int q = q0 + row;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running max of scale*s in log2 units
    float l = 0.f;        // running sum of 2^(scale*s*log2e - m)
    bool ok = true;
    for (int jj = 0; jj < n_kv; ++jj) {
      const int k0 = jj * kBN;
      if (!mbar_wait(bar(C::B_SFULL + (jj & 1)), (jj >> 1) & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_t = tmem + lane_off + C::TM_S + (jj & 1) * 128;
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_t + c * 32, sr[c]);
      tmem_ld_wait(sr[0]);
      reg_fence32(sr[1]);
      reg_fence32(sr[2]);
      reg_fence32(sr[3]);
      // Mask: keys past N (ragged tail) and, on the diagonal tile, keys after q.
      const bool need_mask = (k0 + kBN > p.N) || (p.causal && k0 + kBN - 1 > q0);
      if (need_mask) {
        const int lim = p.causal ? min(p.N - 1, q) : p.N - 1;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (k0 + c * 32 + i > lim) sr[c][i] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sr[c][i]));
      const float m_new = fmaxf(m, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m - m_use);  // 0 on the first tile (m = -inf)
      float rs = 0.f;
      uint32_t pk[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[c][2 * i]), sl2, -m_use));
          const float p1 = ex2(fmaf(__uint_as_float(sr[c][2 * i + 1]), sl2, -m_use));
          rs += p0 + p1;
          pk[c][i] = pack_bf16(p0, p1);
        }
      l = l * alpha + rs;
      m = m_new;
      if (jj > 0) {
        // O holds the sum up to tile jj-1; wait for that PV before rescaling.
        if (!mbar_wait(bar(C::B_ODONE), (jj - 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + C::TM_O + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tmem + lane_off + C::TM_O + c * 32, o);
          }
        }
      }
      // P (bf16) over the first 64 columns of this S buffer.
      {
        uint32_t w0[32], w1[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          w0[i] = pk[0][i];
          w0[16 + i] = pk[1][i];
          w1[i] = pk[2][i];
          w1[16 + i] = pk[3][i];
        }
        tmem_st32(s_t, w0);
        tmem_st32(s_t + 32, w1);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_PFULL + (jj & 1)));
    }
    // Epilogue: O / l and LSE.
    if (ok && mbar_wait(bar(C::B_ODONE), (n_kv - 1) & 1, wc)) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool valid = q < p.N;
      const size_t row_idx = (size_t)bh * p.N + q;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + C::TM_O + c * 32, o);
        tmem_ld_wait(o);
        if (valid) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + row_idx * D + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                   __uint_as_float(o[4 * i + 2]) * inv_l,
                                   __uint_as_float(o[4 * i + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.O) + row_idx * D + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(o[8 * i + 0]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l);
              v.y = pack_bf16(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l);
              v.z = pack_bf16(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l);
              v.w = pack_bf16(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l);
              dst[i] = v;
            }
          }
        }
      }
      if (valid) {
        // LSE = ln(sum_j e^{s_j}) = (m + log2 l) * ln 2, m in log2 units.
        p.LSE[row_idx] = (l > 0.f) ? (m + lg2(l)) * 0.69314718055994531f : -INFINITY;
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
                   const FwdParams& p, cudaStream_t stream) {
  using C = Fwd<D>;
  auto kern = fwd_bf16_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.Hq, p.n_qtiles);
  kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_bf16_smem_bytes(int d) {
  return d == 128 ? Fwd<128>::SMEM_BYTES : Fwd<64>::SMEM_BYTES;
}

cudaError_t launch_fwd_bf16(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const FwdParams& p, cudaStream_t stream) {
  if (d == 128) return launch<128>(tmQ, tmK, tmV, p, stream);
  if (d == 64) return launch<64>(tmQ, tmK, tmV, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
