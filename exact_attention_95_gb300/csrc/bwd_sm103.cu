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
//   bwd_pre     -D_i = -rowsum(dO * O) and -LSE_i * log2(e) into the workspace
//               (stored negated: the main kernel adds them); zeroes the fp32
//               dQ accumulator.
//   bwd_main    one CTA per (batch, kv head, 128-key tile); loops over the G
//               query heads of the group and their 128-row query tiles.  Five
//               tcgen05 products per query tile, all M=128 N=128:
//                 S^T  = K Q^T         -> TMEM region S   (keys on lanes)
//                 dP^T = V dO^T        -> TMEM region DP
//                 dV  += P^T dO        (P^T read from region S as bf16)
//                 dK  += dS^T Q        (dS^T read from region S as bf16)
//                 dQ^T = K^T dS^T      (dS^T from shared memory) -> region DP
//               dK and dV stay in TMEM across the whole group (no atomics);
//               dQ^T is read back and reduce-added (fp32) into the accumulator.
//   bwd_dq      dQ = bf16(scale * accumulator).
//
// Warps of bwd_main (12): 0 TMA producer, 1 TMEM allocator + MMA issuer
// (converged warp, elected lane issues), 2 dQ reducer, 3 idle, 4-7 and 8-11 two math
// warpgroups: thread = key row (TMEM lane), warpgroup h owns query columns
// [64h, 64h + 64) of every tile.  A math thread turns its 64 scores into P
// (bf16, written over the first half of its own score columns), then its 64
// dP values into dS (bf16, over the second half, and into shared memory for
// the dQ product), then reads 64 columns of dQ^T (lane = head-dim index),
// and stages them in shared memory; warp 2 adds each staged half to the
// accumulator with one bulk tensor reduce and then releases the stage.
// Shared memory: K and V tiles, two stages of (Q tile, dO tile, LSE, D).  dS
// for the dQ product is written over the stage's dO tile once dV (the last
// reader of dO) has completed.
#include <algorithm>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBK = 128;  // keys per CTA
constexpr int kBQ = 128;  // query rows per inner tile
constexpr int kMainThreads = 384;
constexpr int kLaunchRegs = 168;  // per-thread registers of a 384-thread CTA
constexpr int kRegsLow = 72;
constexpr int kRegsHigh = 216;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kMainThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;

// MASKED: the block-sparse variant, which keeps a list of (query head, query
// tile) pairs in shared memory.  The dense variant uses that space for a
// dedicated staging buffer of one dQ half (64 query rows), so that a
// stage's Q slot is released as soon as dK has read it and only the dO slot
// waits for a reduce.
template <int D, bool MASKED>
struct Bwd {
  static constexpr bool STAGED = !MASKED;
  static constexpr int CB = D / 64;
  static constexpr int BLK = 128 * 128;  // 128 rows x 128 bytes
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + CB * BLK;
  static constexpr int OFF_STAGE = OFF_V + CB * BLK;
  static constexpr int ST_Q = 0;
  static constexpr int ST_DO = CB * BLK;  // >= 2 blocks: also holds dS^T (128 keys x 128 queries)
  static constexpr int DO_BYTES = (CB < 2 ? 2 : CB) * BLK;
  static constexpr int ST_LSE = ST_DO + DO_BYTES;
  static constexpr int ST_D = ST_LSE + kBQ * 4;
  static constexpr int STAGE_BYTES = (ST_D + kBQ * 4 + 1023) / 1024 * 1024;
  static constexpr int STAGES = 2;
  static constexpr int DQS_BYTES = 64 * D * 4;  // one staged dQ half: 64 query rows x d fp32
  static constexpr int OFF_DQS = OFF_STAGE + STAGES * STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_DQS + (STAGED ? DQS_BYTES : 0);
  static constexpr int B_KVFULL = 0;
  // Each stage has two halves with their own barriers: the Q part (Q tile,
  // -LSE2, -D) and the dO part, released separately by the dQ reducer.
  static constexpr int B_STFULL = 1;                     // STAGES: Q part landed
  static constexpr int B_STFULL_DO = B_STFULL + STAGES;  // STAGES: dO part landed
  static constexpr int B_STEMPTY = B_STFULL_DO + STAGES; // STAGES: Q slot free
  static constexpr int B_STEMPTY_DO = B_STEMPTY + STAGES;  // STAGES: dO slot free
  static constexpr int B_SFULL = B_STEMPTY_DO + STAGES;
  static constexpr int B_DPFULL = B_SFULL + 1;
  static constexpr int B_PFULL = B_DPFULL + 1;
  static constexpr int B_DVDONE = B_PFULL + 1;
  static constexpr int B_DSTMEM = B_DVDONE + 1;  // dS in TMEM (for dK)
  static constexpr int B_DSSMEM = B_DSTMEM + 1;  // dS in shared memory (for dQ)
  static constexpr int B_KVDONE = B_DSSMEM + 1;
  static constexpr int B_DQFULL = B_KVDONE + 1;
  static constexpr int B_DQFREE = B_DQFULL + 1;
  static constexpr int B_DQSTAGED = B_DQFREE + 1;  // 2: one per math warpgroup
  static constexpr int B_DQSFREE = B_DQSTAGED + 2; // dense: the staging buffer has been read
  static constexpr int B_DRAIN = B_DQSFREE + 1;
  static constexpr int NBARS = B_DRAIN + 1;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int OFF_NLIST = OFF_ABORT + 4;   // block-sparse: entries in the list
  static constexpr int OFF_LIST = OFF_NLIST + 4;    // uint32 (g << 16 | query tile) per entry
  // The dense variant has no room for alignment slack: the kernel checks that
  // the dynamic shared memory starts on a 1024-byte boundary.
  static constexpr int SMEM_BYTES = MASKED ? OFF_LIST + 4 * kMaxMaskIters + 1024 : OFF_ABORT + 4;
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB of shared memory per block");
  // TMEM columns
  static constexpr uint32_t TM_DV = 0;
  static constexpr uint32_t TM_DK = D;
  static constexpr uint32_t TM_S = 2 * D;         // 128 columns: S^T, then P | dS (bf16)
  static constexpr uint32_t TM_DP = 2 * D + 128;  // 128 columns: dP^T, then dQ^T
  static constexpr uint32_t IDESC_ST = idesc_bf16(128, kBQ, false, false);
  static constexpr uint32_t IDESC_KV = idesc_bf16(128, D, false, true);
  static constexpr uint32_t IDESC_DQ = idesc_bf16(128, kBQ, true, true);
};

// ------------------------------------------------------------------ preprocess
// One warp per four consecutive rows of the padded row range (four rows never
// straddle two heads: Npad is a multiple of 128): -D, -LSE * log2(e), and
// zeroed accumulator rows.  Rows past N get D = 0 and -LSE2 = -inf
// (probability 0).  All loads of the four rows are issued before any use, so
// each warp keeps 4 x 2 row reads in flight.
constexpr int kRowsPerWarp = 4;
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdParams p) {
  constexpr int EPL = D / 32;  // elements per lane
  using Vec = typename std::conditional<EPL == 4, uint2, uint32_t>::type;
  const long long chunks = (long long)p.B * p.Hq * p.Npad / kRowsPerWarp;
  const int lane = threadIdx.x & 31;
  for (long long c = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < chunks;
       c += ((long long)gridDim.x * blockDim.x) >> 5) {
    const long long r0 = c * kRowsPerWarp;
    const long long bh = r0 / p.Npad;
    const int i0 = (int)(r0 - bh * p.Npad);
    Vec a[kRowsPerWarp], g[kRowsPerWarp];
#pragma unroll
    for (int u = 0; u < kRowsPerWarp; ++u) {
      if (i0 + u < p.N) {
        const size_t off = ((size_t)bh * p.N + i0 + u) * D + lane * EPL;
        a[u] = *reinterpret_cast<const Vec*>(p.O + off);
        g[u] = *reinterpret_cast<const Vec*>(p.dO + off);
      } else {
        a[u] = Vec{};
        g[u] = Vec{};
      }
    }
    // Lane u < 4 fetches the LSE of row u.
    float lse = 0.f;
    if (lane < kRowsPerWarp && i0 + lane < p.N) lse = p.LSE[bh * p.N + i0 + lane];
    float dsum[kRowsPerWarp];
#pragma unroll
    for (int u = 0; u < kRowsPerWarp; ++u) {
      const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a[u]);
      const uint32_t* gw = reinterpret_cast<const uint32_t*>(&g[u]);
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < EPL / 2; ++k) {
        sum += __uint_as_float(aw[k] << 16) * __uint_as_float(gw[k] << 16);
        sum += __uint_as_float(aw[k] & 0xffff0000u) * __uint_as_float(gw[k] & 0xffff0000u);
      }
      dsum[u] = sum;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < kRowsPerWarp; ++u) dsum[u] += __shfl_xor_sync(0xffffffffu, dsum[u], o);
    if (lane < kRowsPerWarp) {
      float mine = dsum[0];
#pragma unroll
      for (int u = 1; u < kRowsPerWarp; ++u)
        if (lane == u) mine = dsum[u];
      p.negD[r0 + lane] = -mine;
      // A row with no kept key (LSE = -inf) gets probability 0, like a padded row.
      p.negLSE2[r0 + lane] = (i0 + lane < p.N && lse != -INFINITY) ? -lse * 1.4426950408889634f : -INFINITY;
    }
    float4* acc = reinterpret_cast<float4*>(p.dQacc + r0 * D);
    for (int k = lane; k < kRowsPerWarp * D / 4; k += 32) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ------------------------------------------------------------------ dQ convert
// dQ = bf16(scale * accumulator): one warp per four consecutive padded rows of
// one head, all four rows' loads issued first.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const BwdParams p) {
  constexpr int V4 = D / 4;  // float4 per row
  const long long chunks = (long long)p.B * p.Hq * p.Npad / kRowsPerWarp;
  const int lane = threadIdx.x & 31;
  for (long long c = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < chunks;
       c += ((long long)gridDim.x * blockDim.x) >> 5) {
    const long long r0 = c * kRowsPerWarp;
    const long long bh = r0 / p.Npad;
    const int i0 = (int)(r0 - bh * p.Npad);
    const float4* src = reinterpret_cast<const float4*>(p.dQacc + r0 * D);
    constexpr int PER_LANE = kRowsPerWarp * V4 / 32;
    float4 v[PER_LANE];
#pragma unroll
    for (int k = 0; k < PER_LANE; ++k) v[k] = src[lane + 32 * k];
#pragma unroll
    for (int k = 0; k < PER_LANE; ++k) {
      const int e = lane + 32 * k;  // float4 index within the four rows
      const int u = e / V4, col = (e - u * V4) * 4;
      if (i0 + u < p.N) {
        uint2 o;
        o.x = pack_bf16(v[k].x * p.scale, v[k].y * p.scale);
        o.y = pack_bf16(v[k].z * p.scale, v[k].w * p.scale);
        *reinterpret_cast<uint2*>(p.dQ + ((size_t)bh * p.N + i0 + u) * D + col) = o;
      }
    }
  }
}

// ------------------------------------------------------------------ main
// P = 2^(s * scale * log2e - LSE2) for the 64 query columns of one math
// warpgroup, two columns per packed FMA (the workspace holds -LSE2): fp32 pairs
// into pv2 (for dS) and bf16 pairs into pk (the dV operand).  With MASK,
// columns c < cmin are zero (keys after the query on a diagonal tile, or a key
// row past N); other tiles skip the per-element test.
template <bool MASK>
__device__ __forceinline__ void bwd_probs(const uint32_t (&sr)[2][32], uint32_t lse_addr, float sl2, int cmin,
                                          uint64_t (&pv2)[32], uint32_t (&pk)[32]) {
  const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll
  for (int c4 = 0; c4 < 16; ++c4) {
    const float4 nl = lds_f4(lse_addr + 16 * c4);  // same address in all lanes
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c = 4 * c4 + 2 * u;
      const uint64_t s2 = f2pack(__uint_as_float(sr[c >> 5][c & 31]), __uint_as_float(sr[c >> 5][(c & 31) + 1]));
      float x0, x1;
      f2unpack(ffma2(s2, sl2x2, u == 0 ? f2pack(nl.x, nl.y) : f2pack(nl.z, nl.w)), x0, x1);
      float p0 = ex2(x0), p1 = ex2(x1);
      if (MASK) {
        if (c < cmin) p0 = 0.f;
        if (c + 1 < cmin) p1 = 0.f;
      }
      pv2[c / 2] = f2pack(p0, p1);
      pk[c / 2] = pack_bf16(p0, p1);
    }
  }
}

constexpr int kDevSmemAlign = 2;  // status: dynamic shared memory not 1024-byte aligned

template <int D, bool MASKED>
__global__ void __launch_bounds__(kMainThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = Bwd<D, MASKED>;
  extern __shared__ uint8_t smem_raw[];
  if (!MASKED && (smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevSmemAlign);
    return;
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V;
  auto stage = [&](int s) -> uint32_t { return sb + C::OFF_STAGE + s * C::STAGE_BYTES; };

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
  const int i0 = p.causal ? (k0 / kBQ) : 0;  // first query tile that sees these keys
  const int per_head = n_q - i0;
  int T = G * per_head;  // inner iterations (>= 1 since k0 < N; may be 0 when masked)
  // Block-sparse: the (query head g, query tile) pairs whose block with this
  // key tile is kept, listed by the otherwise idle warp 3 (ballot compaction).
  constexpr bool masked = MASKED;  // p.bmask != NULL
  uint32_t* const tlist = reinterpret_cast<uint32_t*>(smem + C::OFF_LIST);
  int* const nlist = reinterpret_cast<int*>(smem + C::OFF_NLIST);
  if (masked && warp == 3) {
    int count = 0;
    for (int base = 0; base < T; base += 32) {
      const int t = base + lane;
      bool keep = false;
      uint32_t e = 0;
      if (t < T) {
        const int g = t / per_head, it = i0 + (t - g * per_head);
        const uint8_t* mh = p.bmask + (size_t)(p.bmask_heads == 1 ? 0 : hk * G + g) * n_q * n_q;
        keep = mh[(size_t)it * n_q + jt] != 0;
        e = ((uint32_t)g << 16) | (uint32_t)it;
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      if (keep) tlist[count + __popc(bal & ((1u << lane) - 1u))] = e;
      count += __popc(bal);
    }
    if (lane == 0) *nlist = count;
  }
  auto tile_of = [&](int t, int& g, int& it) {
    if (masked) {
      g = (int)(tlist[t] >> 16);
      it = (int)(tlist[t] & 0xffffu);
    } else {
      g = t / per_head;
      it = i0 + (t - g * per_head);
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KVFULL), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::B_STFULL + s), 1);
      mbar_init(bar(C::B_STFULL_DO + s), 1);
      mbar_init(bar(C::B_STEMPTY + s), 1);     // the dQ reducer (dense: committed after dK)
      mbar_init(bar(C::B_STEMPTY_DO + s), 1);  // arrived by the dQ reducer
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_PFULL), 256);
    mbar_init(bar(C::B_DVDONE), 1);
    mbar_init(bar(C::B_DSTMEM), 256);
    mbar_init(bar(C::B_DSSMEM), 256);
    mbar_init(bar(C::B_KVDONE), 1);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQFREE), 256);
    mbar_init(bar(C::B_DQSTAGED + 0), 128);
    mbar_init(bar(C::B_DQSTAGED + 1), 128);
    mbar_init(bar(C::B_DQSFREE), 1);
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
  if (masked) T = *nlist;

  if (warp < 4) {
    regs_dec<kRegsLow>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::CB * C::BLK);
      if (dcheck(k0 >= 0 && k0 < p.N && bhk >= 0 && bhk < p.B * p.Hkv, p.status))
        for (int cb = 0; cb < C::CB; ++cb) {
          tma_load_3d(sK + cb * C::BLK, &tmK, bar(C::B_KVFULL), cb * 64, k0, bhk);
          tma_load_3d(sV + cb * C::BLK, &tmV, bar(C::B_KVFULL), cb * 64, k0, bhk);
        }
      int tq = 0, tdo = 0;  // Q parts and dO parts issued
      for (int t = 0; t < T; ++t) {
        const int s = t % C::STAGES;
        if (t >= C::STAGES && !mbar_wait(bar(C::B_STEMPTY + s), ((t / C::STAGES) & 1) ^ 1, wc)) break;
        int g, it;
        tile_of(t, g, it);
        const int bhq = b * p.Hq + hk * G + g;
        const uint32_t st = stage(s);
        const uint32_t fb = bar(C::B_STFULL + s);
        mbar_arrive_expect_tx(fb, C::CB * C::BLK + 2 * kBQ * 4);
        const size_t vo = (size_t)bhq * p.Npad + (size_t)it * kBQ;
        if (!dcheck(it >= 0 && it * kBQ < p.N && bhq >= 0 && bhq < p.B * p.Hq &&
                        vo + kBQ <= (size_t)p.B * p.Hq * p.Npad,
                    p.status))
          break;  // (debug builds only: the stage never fills; the waits on it time out)
        for (int cb = 0; cb < C::CB; ++cb)
          tma_load_3d(st + C::ST_Q + cb * C::BLK, &tmQ, fb, cb * 64, it * kBQ, bhq);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                st + C::ST_LSE),
            "l"(p.negLSE2 + vo), "r"(kBQ * 4), "r"(fb)
            : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                st + C::ST_D),
            "l"(p.negD + vo), "r"(kBQ * 4), "r"(fb)
            : "memory");
        tq = t + 1;
        if (t >= C::STAGES && !mbar_wait(bar(C::B_STEMPTY_DO + s), ((t / C::STAGES) & 1) ^ 1, wc)) break;
        const uint32_t fbd = bar(C::B_STFULL_DO + s);
        mbar_arrive_expect_tx(fbd, C::CB * C::BLK);
        for (int cb = 0; cb < C::CB; ++cb)
          tma_load_3d(st + C::ST_DO + cb * C::BLK, &tmdO, fbd, cb * 64, it * kBQ, bhq);
        tdo = t + 1;
      }
      // Before exiting, wait for the copies this thread may still have in flight.
      mbar_wait_drain(bar(C::B_KVFULL), 0, wc);
      for (int k = max(0, tq - C::STAGES); k < tq; ++k)
        mbar_wait_drain(bar(C::B_STFULL + k % C::STAGES), (k / C::STAGES) & 1, wc);
      for (int k = max(0, tdo - C::STAGES); k < tdo; ++k)
        mbar_wait_drain(bar(C::B_STFULL_DO + k % C::STAGES), (k / C::STAGES) & 1, wc);
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp runs this loop (uniform operands); one elected lane issues.
      bool ok = mbar_wait_warp(bar(C::B_KVFULL), 0, wc);
      for (int t = 0; t < T && ok; ++t) {
        const int s = t % C::STAGES;
        const uint32_t st = stage(s);
        const uint32_t qs = st + C::ST_Q, dos = st + C::ST_DO;
        if (!mbar_wait_warp(bar(C::B_STFULL + s), (t / C::STAGES) & 1, wc)) break;
        // Region S is free once dV and dK of the previous tile have completed.
        if (t > 0 && !mbar_wait_warp(bar(C::B_KVDONE), (t - 1) & 1, wc)) break;
        tc_fence_after();
        // S^T = K Q^T (both K-major; 16 head-dim columns per step).
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BLK + (kk & 3) * 32;
          mma_ss_warp(tmem + C::TM_S, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(qs + off, 16, 1024),
                      C::IDESC_ST, kk > 0 ? 1u : 0u);
        }
        tc_commit_warp(bar(C::B_SFULL));
        // Region DP is free once the previous dQ^T has been read back.
        if (t > 0 && !mbar_wait_warp(bar(C::B_DQFREE), (t - 1) & 1, wc)) break;
        if (!mbar_wait_warp(bar(C::B_STFULL_DO + s), (t / C::STAGES) & 1, wc)) break;
        tc_fence_after();
        // dP^T = V dO^T.
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BLK + (kk & 3) * 32;
          mma_ss_warp(tmem + C::TM_DP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(dos + off, 16, 1024),
                      C::IDESC_ST, kk > 0 ? 1u : 0u);
        }
        tc_commit_warp(bar(C::B_DPFULL));
        // dV += P^T dO: 16 queries per step; P of query columns [64h, 64h+64)
        // sits in region S columns [64h, 64h+32) as packed bf16 pairs.
        if (!mbar_wait_warp(bar(C::B_PFULL), t & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_ts_warp(tmem + C::TM_DV, tmem + C::TM_S + (kk >> 2) * 64 + (kk & 3) * 8,
                      sdesc_sw128(dos + kk * 2048, C::BLK, 1024), C::IDESC_KV,
                      (t > 0 || kk > 0) ? 1u : 0u);
        tc_commit_warp(bar(C::B_DVDONE));
        // dK += dS^T Q (dS in region S columns [64h+32, 64h+64)).
        if (!mbar_wait_warp(bar(C::B_DSTMEM), t & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_ts_warp(tmem + C::TM_DK, tmem + C::TM_S + (kk >> 2) * 64 + 32 + (kk & 3) * 8,
                      sdesc_sw128(qs + kk * 2048, C::BLK, 1024), C::IDESC_KV,
                      (t > 0 || kk > 0) ? 1u : 0u);
        tc_commit_warp(bar(C::B_KVDONE));
        // Dense: dK is the last reader of the stage's Q part (Q, -LSE2, -D; the
        // math warps read -LSE2 and -D before dS reached TMEM), so the
        // producer may refill it once dK completes.
        if (C::STAGED) tc_commit_warp(bar(C::B_STEMPTY + s));
        if (!mbar_wait_warp(bar(C::B_DSSMEM), t & 1, wc)) break;
        tc_fence_after();
        // dQ^T = K^T dS^T: A = K as MN-major [d x keys], B = dS^T in the dO
        // slot, MN-major [keys x queries] (two 64-query blocks).  For d = 64
        // the product still has M = 128; lanes 64..127 read the V tile as
        // filler and are discarded.
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_ss_warp(tmem + C::TM_DP, sdesc_sw128(sK + kk * 2048, C::BLK, 1024),
                      sdesc_sw128(dos + kk * 2048, C::BLK, 1024), C::IDESC_DQ, kk > 0 ? 1u : 0u);
        tc_commit_warp(bar(C::B_DQFULL));
      }
      tc_commit_warp(bar(C::B_DRAIN));
      mbar_wait_drain_warp(bar(C::B_DRAIN), 0, wc);
    } else if (warp == 2 && lane == 0) {
      // ---------------------------------------------------------- dQ reducer
      // Adds each staged dQ half-tile to the accumulator with one bulk tensor
      // reduce and releases the stage once the reduces have read it.
      for (int t = 0; t < T; ++t) {
        const int s = t % C::STAGES;
        int g, it;
        tile_of(t, g, it);
        const int bhq = b * p.Hq + hk * G + g;
        const uint32_t st = stage(s);
        const int row0 = (int)((size_t)bhq * p.Npad + (size_t)it * kBQ);
        if (!dcheck(row0 >= 0 && (size_t)row0 + kBQ <= (size_t)p.B * p.Hq * p.Npad, p.status)) break;
        if (C::STAGED) {
          // The half in the dO slot first (the next loads wait for it), then
          // the half in the staging buffer.
          if (!mbar_wait(bar(C::B_DQSTAGED + 1), t & 1, wc)) break;
          tma_reduce_add_2d(&tmDQ, st + C::ST_DO, 0, row0 + 64);
          bulk_commit_group();
          if (!mbar_wait(bar(C::B_DQSTAGED + 0), t & 1, wc)) break;
          tma_reduce_add_2d(&tmDQ, sb + C::OFF_DQS, 0, row0);
          bulk_commit_group();
          bulk_wait_read1();
          mbar_arrive(bar(C::B_STEMPTY_DO + s));
          bulk_wait_read0();
          mbar_arrive(bar(C::B_DQSFREE));
          continue;
        }
        bool ok = true;
        for (int h = 0; h < 2 && ok; ++h) {
          if (!mbar_wait(bar(C::B_DQSTAGED + h), t & 1, wc)) {
            ok = false;
            break;
          }
          tma_reduce_add_2d(&tmDQ, st + (h == 0 ? C::ST_Q : C::ST_DO), 0, row0 + 64 * h);
          bulk_commit_group();
        }
        if (!ok) break;
        bulk_wait_read1();  // the first half (Q slot) has been read
        mbar_arrive(bar(C::B_STEMPTY + s));
        bulk_wait_read0();
        mbar_arrive(bar(C::B_STEMPTY_DO + s));
      }
      bulk_wait0();
    }
  } else {
    regs_inc<kRegsHigh>();
    // ------------------------------------------------------------ math warpgroups
    const int h = (warp - 4) >> 2;  // query-column half of this warpgroup
    const int quad = warp & 3;
    const int kr = quad * 32 + lane;  // key row (TMEM lane) of the S / dP regions
    const int key = k0 + kr;
    const bool key_ok = key < p.N;
    const int dcol = kr;  // head-dim index (TMEM lane) of the dQ^T region
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S + 64 * h;
    const uint32_t tDP = tmem + lane_off + C::TM_DP + 64 * h;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t % C::STAGES;
      int g, it;
      tile_of(t, g, it);
      const int qh0 = it * kBQ + 64 * h;  // first query column of this half
      const int bhq = b * p.Hq + hk * G + g;
      const uint32_t st = stage(s);
      if (!mbar_wait(bar(C::B_STFULL + s), (t / C::STAGES) & 1, wc) ||
          !mbar_wait(bar(C::B_SFULL), t & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // ---- P for this warpgroup's 64 query columns.
      uint32_t sr[2][32];
      tmem_ld32(tS, sr[0]);
      tmem_ld32(tS + 32, sr[1]);
      tmem_ld_wait(sr[0]);
      reg_fence32(sr[1]);
      uint64_t pv2[32];  // P, column pairs
      uint32_t pk[32];
      const uint32_t lse_addr = st + C::ST_LSE + 4 * 64 * h;
      // Tile-uniform test: a ragged key tile, or a causal tile that crosses the diagonal.
      if (k0 + kBK > p.N || (p.causal && qh0 < k0 + kBK - 1)) {
        const int cmin = !key_ok ? 64 : (p.causal ? max(0, key - qh0) : 0);
        bwd_probs<true>(sr, lse_addr, sl2, cmin, pv2, pk);
      } else {
        bwd_probs<false>(sr, lse_addr, sl2, 0, pv2, pk);
      }
      tmem_st32(tS, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_PFULL));
      // ---- dS = P (dP - D), 32 columns at a time (the workspace holds -D).
      if (!mbar_wait(bar(C::B_DPFULL), t & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t dr[32];
        tmem_ld32(tDP + 32 * half, dr);
        tmem_ld_wait(dr);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 nd = lds_f4(st + C::ST_D + 4 * (64 * h + 32 * half + 4 * c4));
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int cp = 16 * half + 2 * c4 + u;  // column pair index
            const uint64_t dp2 = f2pack(__uint_as_float(dr[4 * c4 + 2 * u]), __uint_as_float(dr[4 * c4 + 2 * u + 1]));
            const uint64_t ds2 = fmul2(pv2[cp], fadd2(dp2, u == 0 ? f2pack(nd.x, nd.y) : f2pack(nd.z, nd.w)));
            float d0, d1;
            f2unpack(ds2, d0, d1);
            pk[cp] = pack_bf16(d0, d1);
          }
        }
      }
      tmem_st32(tS + 32, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_DSTMEM));
      // dS^T rows into the dO slot (dV, its last reader, must be complete):
      // block h holds query columns [64h, 64h+64); row kr is 128 bytes with
      // the 16-byte chunk c stored at chunk position c ^ (kr & 7).
      if (!mbar_wait(bar(C::B_DVDONE), t & 1, wc)) {
        ok = false;
        break;
      }
      const uint32_t dsrow = st + C::ST_DO + h * C::BLK + kr * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        sts_u4(dsrow + ((c ^ (kr & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_async_smem();
      mbar_arrive(bar(C::B_DSSMEM));
      // ---- dQ^T readback: 64 query columns of head-dim row dcol.
      if (!mbar_wait(bar(C::B_DQFULL), t & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t qr[2][32];
      tmem_ld32(tDP, qr[0]);
      tmem_ld32(tDP + 32, qr[1]);
      tmem_ld_wait(qr[0]);
      reg_fence32(qr[1]);
      tc_fence_before();
      mbar_arrive(bar(C::B_DQFREE));
      // Stage this half of dQ (64 query rows x d, fp32, row-major) in shared
      // memory -- warpgroup 1 over the dO slot (free once dQ^T has completed),
      // warpgroup 0 over the staging buffer once the previous tile's reduce
      // has read it (the masked variant: over the Q slot) -- and add it to
      // the accumulator with one bulk tensor reduce.
      const uint32_t qstage = h == 1 ? st + C::ST_DO : C::STAGED ? sb + C::OFF_DQS : st + C::ST_Q;
      if (C::STAGED && h == 0 && t > 0 && !mbar_wait(bar(C::B_DQSFREE), (t - 1) & 1, wc)) {
        ok = false;
        break;
      }
      if (dcol < D) {
#pragma unroll
        for (int c = 0; c < 64; ++c) sts_f32(qstage + (c * D + dcol) * 4, __uint_as_float(qr[c >> 5][c & 31]));
      }
      fence_async_smem();
      mbar_arrive(bar(C::B_DQSTAGED + h));
    }
    // Epilogue: dV and scale * dK rows of this key tile; warpgroup h writes
    // head-dim columns [h*D/2, (h+1)*D/2).
    // (A key tile that no kept block reaches writes zero dK and dV.)
    const bool have = T > 0;
    if (ok && (!have || mbar_wait(bar(C::B_KVDONE), (T - 1) & 1, wc))) {
      if (have) tc_fence_after();
      const size_t row = (size_t)bhk * p.N + key;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        uint16_t* dst = (which == 0 ? p.dV : p.dK) + row * D;
        const float mul = which == 0 ? 1.f : p.scale;
        const uint32_t base = tmem + lane_off + (which == 0 ? C::TM_DV : C::TM_DK);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const int col = h * (D / 2) + 32 * c;
          uint32_t o[32];
          if (have) {
            tmem_ld32(base + col, o);
            tmem_ld_wait(o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
          if (key_ok && dcheck(row < (size_t)p.B * p.Hkv * p.N, p.status)) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + col);
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
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool MASKED>
cudaError_t launch_main(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const CUtensorMap& tmdO, const CUtensorMap& tmDQ, const BwdParams& p,
                        cudaStream_t stream) {
  using C = Bwd<D, MASKED>;
  auto kern = bwd_main_kernel<D, MASKED>;
  // setmaxnreg moves registers inside the launch allocation; refuse to launch
  // if the compiler gave the kernel a different per-thread count than assumed.
  static int regs = -1;  // one per instantiation
  cudaError_t e;
  if (regs < 0) {
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    regs = fa.numRegs;
  }
  if (regs != kLaunchRegs) return cudaErrorInvalidKernelImage;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.Hkv * ((p.N + kBK - 1) / kBK));
  kern<<<grid, kMainThreads, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, tmdO, tmDQ, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                   const CUtensorMap& tmdO, const CUtensorMap& tmDQ, const BwdParams& p,
                   unsigned stages, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = cudaSuccess;
  if (stages & kBwdPre) {
    const long long warps = (long long)p.B * p.Hq * p.Npad / kRowsPerWarp;
    const int pre_blocks = (int)std::min<long long>((warps + 7) / 8, (long long)sms * 8);
    bwd_pre_kernel<D><<<pre_blocks, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (stages & kBwdMain) {
    e = p.bmask ? launch_main<D, true>(tmQ, tmK, tmV, tmdO, tmDQ, p, stream)
                : launch_main<D, false>(tmQ, tmK, tmV, tmdO, tmDQ, p, stream);
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdConvert) {
    const long long warps = (long long)p.B * p.Hq * p.Npad / kRowsPerWarp;
    const int cv_blocks = (int)std::min<long long>((warps + 7) / 8, (long long)sms * 8);
    bwd_dq_kernel<D><<<cv_blocks, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return e;
}

}  // namespace

int bwd_row_padding() { return kBQ; }

size_t bwd_workspace_bytes(int B, int Hq, int N, int d) {
  const size_t Npad = (size_t)(N + kBQ - 1) / kBQ * kBQ;
  const size_t rows = (size_t)B * Hq * Npad;
  return (rows * d * 4 + 255) / 256 * 256 + 2 * ((rows * 4 + 255) / 256 * 256);
}

cudaError_t launch_bwd_bf16(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmDQ,
                            const BwdParams& p, unsigned stages, cudaStream_t stream) {
  if (d == 128) return launch<128>(tmQ, tmK, tmV, tmdO, tmDQ, p, stages, stream);
  if (d == 64) return launch<64>(tmQ, tmK, tmV, tmdO, tmDQ, p, stages, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
