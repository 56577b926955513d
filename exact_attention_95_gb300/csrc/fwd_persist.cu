// fwd_persist.cu -- persistent form of the two-tile forward (dense, bf16).
//
// Same computation as fwd_sm103.cu's two-tile kernel: per 128-row query tile
// the online (m, l, O) merge of "LLM 注意力与计算内核精读笔记 · 02
// FlashAttention" §5 over the K/V tiles, 1/l applied once at the end
// ("从Online-Softmax到FlashAttention V1/V2/V3", 0x05), causal tiles past the
// diagonal never visited and GQA by head indexing (0x09).
//
// What differs is the life of a CTA.  One CTA runs per SM and walks work
// items -- (key split, head, pair of 128-row query tiles), in the order of
// the one-CTA-per-item grid: heaviest pairs first within groups of heads --
// taken from a global counter, so that an SM that finishes a light item
// takes the next one at once (longest-first list scheduling).  TMEM, the
// mbarriers and the tensor-map prefetch are set up once per CTA; the
// producer loads the next item's Q and K/V tiles while the current item
// computes; and the next item's first Q K^T is issued right behind the
// current item's last P V, so a pair's epilogue (O / l and LSE read out of
// TMEM and stored) overlaps the next pair's first products.
//
// Roles (12 warps):
//   warp 0      producer: takes items from the global counter into a
//               two-entry ring in shared memory, loads Q tile 0, K_0, Q tile
//               1, then K_{j+1} ahead of V_j through the K/V ring.
//   warp 1      TMEM owner; MMA issuer of query tile 0 (converged warp,
//               elected lane).
//   warp 2      MMA issuer of query tile 1.  Issuing an M = N = 128 product
//               takes a warp about as long as the tensor pipe takes to run
//               it, so with one issuing warp every wait of that warp left the
//               pipe idle; two warps keep it fed while either one waits.
//   warps 4-7   softmax and epilogue of query tile 0, warps 8-11 of tile 1.
// Every phase counter (ring slots, S buffer, P and O hand-offs) runs on
// across items.  The counter pair of the launch is reset by the last CTA to
// finish, so the next launch on the same counter starts at zero.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 72;
constexpr int kRegsHigh = 216;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 16.0f;  // log2 units, as in the one-CTA-per-item kernel

template <int D>
struct FwdP {
  static constexpr int CB = D / 64;
  static constexpr int BLOCK_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = CB * BLOCK_BYTES;
  static constexpr int STAGES = D == 128 ? 4 : 8;
  static constexpr int IR = 2;  // item ring entries
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TILE_BYTES;
  static constexpr int B_QFULL = 0;                  // 2: Q tile t landed
  static constexpr int B_QEMPTY = B_QFULL + 2;       // 2: Q tile t read by its last S
  static constexpr int B_KVFULL = B_QEMPTY + 2;
  static constexpr int B_KVEMPTY = B_KVFULL + STAGES;
  static constexpr int B_SFULL = B_KVEMPTY + STAGES;  // 2
  static constexpr int B_SREAD = B_SFULL + 2;         // 2: S_t read out of the S buffer
  static constexpr int B_PFULL = B_SREAD + 2;         // 2
  static constexpr int B_ODONE = B_PFULL + 2;         // 2
  static constexpr int B_ITFULL = B_ODONE + 2;        // IR: ring entry written
  static constexpr int B_ITEMPTY = B_ITFULL + IR;     // IR: ring entry read by every consumer warp
  static constexpr int B_DRAIN = B_ITEMPTY + IR;     // 2: one per issuing warp
  static constexpr int NBARS = B_DRAIN + 2;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int OFF_RING = OFF_ABORT + 4;
  static constexpr int RING_INTS = 8;                  // one decoded item per entry
  // Epilogue staging: per softmax warp, its 32 rows x 64 columns of bf16 O.
  static constexpr int EPI_WARP_BYTES = 32 * 128;
  static constexpr int OFF_EPI = (OFF_RING + 4 * RING_INTS * IR + 127) / 128 * 128;
  static constexpr int SMEM_BYTES = OFF_EPI + 8 * EPI_WARP_BYTES + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB of shared memory per block");
  static constexpr int CONSUMER_WARPS = 2 + 8;  // the two MMA warps and the softmax warps
  static constexpr uint32_t IDESC_S = idesc_bf16(kBM, kBN, false, false);
  static constexpr uint32_t IDESC_O = idesc_bf16(kBM, D, false, true);
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_P = 128;
  static constexpr uint32_t TM_O = 256;
};

// A work item: key split, grid head and tile pair, decoded from its index
// exactly as the one-CTA-per-item kernel decodes blockIdx.x.
struct FwdItem {
  int bh;     // grid head (b * Hq + h)
  int q0;     // first query row of the pair
  int kt0;    // first K/V tile of the split
  int n_kv;   // K/V tiles visited (0: the split lies wholly right of the diagonal)
  int bh_kv;  // K/V head
  int split;
};

__device__ __forceinline__ FwdItem fwd_item(int k, const FwdParams& p) {
  FwdItem w;
  w.split = k % p.n_splits;
  int rank;
  grouped_order(k / p.n_splits, p.heads, p.n_pairs, p.head_group, w.bh, rank);
  const int pair = p.n_pairs - 1 - rank;
  w.q0 = pair * 2 * kBM;
  const int b = w.bh / p.Hq;
  const int h = w.bh - b * p.Hq;
  w.bh_kv = p.packed ? w.bh : b * p.Hkv + h / (p.Hq / p.Hkv);
  w.kt0 = w.split * p.tiles_per_split;
  int kt_end = min(w.kt0 + p.tiles_per_split, (p.Nk + kBN - 1) / kBN);
  if (p.causal) {
    const int k_last = (p.packed ? p.N : min(w.q0 + 2 * kBM, p.N)) - 1 + p.kv_off;
    kt_end = k_last < 0 ? 0 : min(kt_end, k_last / kBN + 1);
  }
  w.n_kv = max(0, kt_end - w.kt0);
  return w;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdP<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q;
  const uint32_t sKV = sb + C::OFF_KV;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_RING);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_QFULL + t), 1);
      mbar_init(bar(C::B_QEMPTY + t), 1);
      mbar_init(bar(C::B_SFULL + t), 1);
      mbar_init(bar(C::B_PFULL + t), 4);  // one arrival per softmax warp
      mbar_init(bar(C::B_ODONE + t), 1);
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::B_KVFULL + s), 1);
      mbar_init(bar(C::B_KVEMPTY + s), 2);  // a K or V tile is read by both tiles' products
    }
    for (int r = 0; r < C::IR; ++r) {
      mbar_init(bar(C::B_ITFULL + r), 1);
      mbar_init(bar(C::B_ITEMPTY + r), C::CONSUMER_WARPS);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_SREAD + t), 4);  // one arrival per softmax warp of tile t
      mbar_init(bar(C::B_DRAIN + t), 1);
    }
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

  // Ring entry r: item index (-1: none left), then its decoded fields.  A
  // consumer warp waits for the entry of its item `it`, reads the fields
  // whenever it needs them, and releases the entry (one arrival per warp)
  // when it is done with the item, so the producer runs at most one item
  // ahead of the slowest consumer.
  enum { R_K = 0, R_BH, R_Q0, R_KT0, R_NKV, R_BHKV, R_SPLIT };
  auto entry = [&](int it) -> volatile int* { return ring + (it % C::IR) * C::RING_INTS; };
  auto wait_item = [&](int it) -> bool {
    return mbar_wait_warp(bar(C::B_ITFULL + it % C::IR), (it / C::IR) & 1, wc);
  };
  auto release_item = [&](int it) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(C::B_ITEMPTY + it % C::IR));
  };

  if (warp < 4) {
    regs_dec<kRegsLow>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int li = 0;             // K/V loads issued (ring position)
      int qi[2] = {0, 0};     // Q tile loads issued, per tile (one per item with keys)
      bool ok = true;
      auto load_q = [&](int t, const FwdItem& w) -> bool {
        if (qi[t] > 0 && !mbar_wait(bar(C::B_QEMPTY + t), (qi[t] - 1) & 1, wc)) return false;
        mbar_arrive_expect_tx(bar(C::B_QFULL + t), C::TILE_BYTES);
        const int r0 = w.q0 + t * kBM;  // may start past the last row (zero fill) in a ragged last pair
        if (dcheck(r0 >= 0 && r0 < p.n_pairs * 2 * kBM && w.bh >= 0 && w.bh < p.heads, p.status))
          for (int cb = 0; cb < C::CB; ++cb)
            tma_load_3d(sQ + t * C::TILE_BYTES + cb * C::BLOCK_BYTES, &tmQ, bar(C::B_QFULL + t), cb * 64, r0,
                        w.bh);
        ++qi[t];
        return true;
      };
      auto load_kv = [&](bool v, int kt, int bh_kv) -> bool {
        const int s = li % C::STAGES;
        if (li >= C::STAGES && !mbar_wait(bar(C::B_KVEMPTY + s), ((li / C::STAGES) & 1) ^ 1, wc))
          return false;
        mbar_arrive_expect_tx(bar(C::B_KVFULL + s), C::TILE_BYTES);
        const CUtensorMap* m = v ? &tmV : &tmK;
        const int kv_heads = p.packed ? p.heads : p.B * p.Hkv;
        if (dcheck(kt >= 0 && kt * kBN < p.Nk && bh_kv >= 0 && bh_kv < kv_heads, p.status))
          for (int cb = 0; cb < C::CB; ++cb)
            tma_load_3d(sKV + s * C::TILE_BYTES + cb * C::BLOCK_BYTES, m, bar(C::B_KVFULL + s), cb * 64,
                        kt * kBN, bh_kv);
        ++li;
        return true;
      };
      for (int it = 0; ok; ++it) {
        const int r = it % C::IR;
        if (it >= C::IR && !mbar_wait(bar(C::B_ITEMPTY + r), ((it / C::IR) - 1) & 1, wc)) break;
        int k = (int)atomicAdd(p.sched, 1u);
        if (k >= p.n_items) k = -1;
        volatile int* e = entry(it);
        const FwdItem w = fwd_item(k < 0 ? 0 : k, p);
        e[R_K] = k;
        e[R_BH] = w.bh;
        e[R_Q0] = w.q0;
        e[R_KT0] = w.kt0;
        e[R_NKV] = w.n_kv;
        e[R_BHKV] = w.bh_kv;
        e[R_SPLIT] = w.split;
        mbar_arrive(bar(C::B_ITFULL + r));
        if (k < 0) {
          // No item left: a merge launched behind this kernel may start (it
          // waits for this kernel's completion before reading).
          griddep_launch_dependents();
          break;
        }
        const int n = w.n_kv;
        if (n == 0) continue;
        // Use order: Q_0, K_0, Q_1, then K_{j+1} ahead of V_j.
        ok = load_q(0, w) && load_kv(false, w.kt0, w.bh_kv) && load_q(1, w);
        for (int u = 1; u < 2 * n && ok; ++u) {
          int j;
          bool v;
          if (n == 1) {
            v = true;
            j = 0;
          } else if (u == 2 * n - 1) {
            v = true;
            j = n - 1;
          } else {
            v = (u % 2 == 0);
            j = v ? u / 2 - 1 : (u + 1) / 2;
          }
          ok = load_kv(v, w.kt0 + j, w.bh_kv);
        }
      }
      // Drain: every issued copy must land before the CTA may exit (at most
      // one Q copy per tile is in flight: the next waits for QEMPTY).
      for (int t = 0; t < 2; ++t)
        if (qi[t] > 0) mbar_wait_drain(bar(C::B_QFULL + t), (qi[t] - 1) & 1, wc);
      for (int k = max(0, li - C::STAGES); k < li; ++k)
        mbar_wait_drain(bar(C::B_KVFULL + k % C::STAGES), (k / C::STAGES) & 1, wc);
    } else if (warp == 1 || warp == 2) {
      // ---------------------------------------------------------- MMA issuers
      // Warp 1 issues query tile 0's products, warp 2 tile 1's.  A warp
      // needs about as long to issue one M = N = 128 product as the tensor
      // pipe needs to run it, so one issuing warp keeps the pipe busy only
      // if it never waits; with two, either warp's products keep the pipe
      // busy while the other waits.  Per tile: S_t(0), then for each j,
      // S_t(j+1) ahead of P_t(j) V_j.  The one S buffer still alternates
      // S_0(j), S_1(j), S_0(j+1): tile 1's S(j) waits until tile 0 has read
      // S_0(j), tile 0's S(j+1) until tile 1 has read S_1(j).
      const int t = warp - 1;
      int li0 = 0;        // ring position of the current item's first K/V load
      int qn = 0;         // items with Q loaded so far
      int ns = 0;         // S products of this tile issued so far
      int pf = 0;         // PFULL_t completions waited for
      bool ok = true;
      for (int it = 0; ok; ++it) {
        if (!wait_item(it)) break;
        const int k = entry(it)[R_K];
        const int n = entry(it)[R_NKV];
        release_item(it);
        if (k < 0) break;
        if (n == 0) continue;
        auto k_li = [&](int j) -> int { return li0 + (j == 0 ? 0 : 2 * j - 1); };
        auto v_li = [&](int j) -> int { return li0 + (j == n - 1 ? 2 * n - 1 : 2 * j + 2); };
        auto wait_kv = [&](int li) -> bool {
          if (!mbar_wait_warp(bar(C::B_KVFULL + li % C::STAGES), (li / C::STAGES) & 1, wc)) return false;
          tc_fence_after();
          return true;
        };
        // The S buffer is free for this tile's next S once the other tile
        // has read the S issued before it: tile 1's ns-th S follows tile 0's
        // ns-th, tile 0's ns-th follows tile 1's (ns - 1)-th.
        auto wait_sbuf = [&]() -> bool {
          if (t == 0 && ns == 0) return true;
          const int phase = t == 0 ? ns - 1 : ns;
          if (!mbar_wait_warp(bar(C::B_SREAD + (t ^ 1)), phase & 1, wc)) return false;
          tc_fence_after();
          return true;
        };
        // Descriptors of later K steps are the first one plus the byte
        // offset / 16 in the address field (shared addresses stay below
        // 256 KB, so the 14-bit field does not carry).
        // (The empty asm keeps the compiler from hoisting the CTA-constant Q
        // descriptors of every K step out of the item loop: registers the
        // 72-register issuing warps do not have.)
        auto issue_s = [&](int j) {
          uint64_t qd = sdesc_sw128(sQ + t * C::TILE_BYTES, 16, 1024);
          asm volatile("" : "+l"(qd));
          const uint64_t kd = sdesc_sw128(sKV + (k_li(j) % C::STAGES) * C::TILE_BYTES, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off16 = ((kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32) >> 4;
            mma_ss_warp(tmem + C::TM_S, qd + off16, kd + off16, C::IDESC_S, kk > 0 ? 1u : 0u);
          }
          tc_commit_warp(bar(C::B_SFULL + t));
          if (j == n - 1) tc_commit_warp(bar(C::B_QEMPTY + t));        // last reader of Q_t
          tc_commit_warp(bar(C::B_KVEMPTY + k_li(j) % C::STAGES));    // one of K_j's two readers
          ++ns;
        };
        auto issue_pv = [&](int j) {
          const uint64_t vd = sdesc_sw128(sKV + (v_li(j) % C::STAGES) * C::TILE_BYTES, C::BLOCK_BYTES, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_warp(tmem + C::TM_O + t * D, tmem + C::TM_P + t * 64 + kk * 8, vd + (kk * 2048 >> 4),
                        C::IDESC_O, (kk > 0 || j > 0) ? 1u : 0u);
          tc_commit_warp(bar(C::B_ODONE + t));
          tc_commit_warp(bar(C::B_KVEMPTY + v_li(j) % C::STAGES));    // one of V_j's two readers
        };
        auto wait_p = [&]() -> bool {
          const bool r = mbar_wait_warp(bar(C::B_PFULL + t), pf & 1, wc);
          ++pf;
          if (r) tc_fence_after();
          return r;
        };
        ok = wait_sbuf() && mbar_wait_warp(bar(C::B_QFULL + t), qn & 1, wc) && wait_kv(k_li(0));
        if (ok) issue_s(0);
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n) {
            if (!wait_sbuf() || !wait_kv(k_li(j + 1))) {
              ok = false;
              break;
            }
            issue_s(j + 1);
          }
          if (!wait_kv(v_li(j)) || !wait_p()) {
            ok = false;
            break;
          }
          issue_pv(j);
        }
        li0 += 2 * n;
        ++qn;
      }
      // Drain: all MMAs of this warp complete before TMEM is released.
      tc_commit_warp(bar(C::B_DRAIN + t));
      mbar_wait_drain_warp(bar(C::B_DRAIN + t), 0, wc);
    }
  } else {
    regs_inc<kRegsHigh>();
    // ------------------------------------------------------------ softmax + epilogue
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_t = tmem + lane_off + C::TM_S;
    const uint32_t p_t = tmem + lane_off + C::TM_P + t * 64;
    const uint32_t o_t = tmem + lane_off + C::TM_O + t * D;
    const uint32_t sEpi = sb + C::OFF_EPI + (warp - 4) * C::EPI_WARP_BYTES;
    const float sl2 = p.scale_log2;
    // S tiles of this warpgroup completed so far (SFULL_t phases).  Each
    // tile but an item's first waits for the previous P_t V, and the
    // epilogue for the last: the ODONE_t phase waited for at step j > 0 is
    // sg - 2 (after the increment below), in the epilogue sg - 1.
    int sg = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      if (!wait_item(it)) break;
      volatile int* e = entry(it);
      if (e[R_K] < 0) {
        release_item(it);
        break;
      }
      const int n = e[R_NKV];
      const int qt0 = e[R_Q0] + t * kBM;
      const int q = qt0 + row;
      const int qc = p.packed ? q % p.N : q;
      const int qc0 = p.packed ? 0 : qt0;
      float m = -INFINITY;
      float l = 0.f;
      float corr = 0.f;
      for (int j = 0; j < n; ++j) {
        const int k0 = (e[R_KT0] + j) * kBN;
        if (!mbar_wait_warp(bar(C::B_SFULL + t), sg & 1, wc)) {
          ok = false;
          break;
        }
        ++sg;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_t + c * 32, sr[c]);
        tmem_ld_wait(sr[0]);
        reg_fence32(sr[1]);
        reg_fence32(sr[2]);
        reg_fence32(sr[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_SREAD + t));
        if ((k0 + kBN > p.Nk) || (p.causal && k0 + kBN - 1 > qc0 + p.kv_off)) {
          const int lim = p.causal ? min(p.Nk - 1, qc + p.kv_off) : p.Nk - 1;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (k0 + c * 32 + i > lim) sr[c][i] = __float_as_uint(-INFINITY);
        }
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            mp[i & 7] = fmax3(mp[i & 7], __uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1]));
        const float mraw = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                 fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        const float mx = mraw * sl2;
        const bool move = mx > m + kRescaleThreshold;
        float alpha = 1.f;
        if (move) {
          alpha = ex2(m - mx);
          m = mx;
          l *= alpha;
          corr *= alpha;
        }
        const float m_use = (m == -INFINITY) ? 0.f : m;
        {
          const float pmax = ex2(fmaf(mraw, sl2, -m_use));
          corr += pmax - __uint_as_float(pack_bf16(pmax, pmax) & 0xffff0000u);
        }
        uint64_t rs2[4] = {0, 0, 0, 0};
        const uint64_t sl2x2 = f2pack(sl2, sl2);
        const uint64_t negm2 = f2pack(-m_use, -m_use);
        uint32_t wv[2][32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2unpack(ffma2(f2pack(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), sl2x2, negm2),
                     x0, x1);
            const float p0 = ex2(x0);
            const float p1 = ex2(x1);
            rs2[i & 3] = fadd2(rs2[i & 3], f2pack(p0, p1));
            wv[c >> 1][(c & 1) * 16 + i] = pack_bf16(p0, p1);
          }
        {
          float a0, a1;
          f2unpack(fadd2(fadd2(rs2[0], rs2[1]), fadd2(rs2[2], rs2[3])), a0, a1);
          l += a0 + a1;
        }
        if (j > 0) {
          // The previous P_t V of this item must be complete: it reads the
          // P_t columns written below, and O_t may be rescaled.
          if (!mbar_wait_warp(bar(C::B_ODONE + t), sg & 1, wc)) {  // phase sg - 2
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, move)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(o_t + c * 32, sr[c]);
            tmem_ld_wait(sr[0]);
#pragma unroll
            for (int c = 1; c < D / 32; ++c) reg_fence32(sr[c]);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
#pragma unroll
              for (int i = 0; i < 32; ++i) sr[c][i] = __float_as_uint(__uint_as_float(sr[c][i]) * alpha);
              tmem_st32(o_t + c * 32, sr[c]);
            }
          }
        }
        // (j == 0: the previous item's last P_t V completed before its
        // epilogue read O_t, so the P_t columns are free.)
        tmem_st32(p_t, wv[0]);
        tmem_st32(p_t + 32, wv[1]);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_PFULL + t));
      }
      if (!ok) break;
      // Epilogue: O / (l - corr) and LSE (O = 0, LSE = -inf when no key was in range).
      if (n > 0) {
        if (!mbar_wait_warp(bar(C::B_ODONE + t), (sg - 1) & 1, wc)) break;
        tc_fence_after();
      }
      const int split = e[R_SPLIT];
      float* const o_out = p.out_f32 ? static_cast<float*>(p.O) + split * p.o_split_stride : nullptr;
      uint16_t* const o_out16 = p.out_f32 ? nullptr : static_cast<uint16_t*>(p.O);
      const float lo = l - corr;
      const float inv_l = lo > 0.f ? 1.f / lo : 0.f;
      const int bh = e[R_BH];
      const bool bh_ok = dcheck(bh >= 0 && bh < p.heads && split >= 0 && split < p.n_splits, p.status);
      const bool valid = q < p.rows && bh_ok;
      const size_t row_idx = (size_t)bh * p.rows + q;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(o_t + c * 32, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (valid) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(o_out + row_idx * D + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                   __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
          } else {
            epi_stage32(sEpi, lane, c, o, inv_l);
          }
        }
        // bf16: after each 64-column half, the warp stores its 32 rows.
        if (!p.out_f32 && (c & 1))
          epi_store_half(sEpi, lane, c >> 1, o_out16, (size_t)bh * p.rows + qt0 + quad * 32, D,
                         bh_ok ? p.rows - (qt0 + quad * 32) : 0);
      }
      if (valid) {
        float* const lse_out = p.LSE + split * p.lse_split_stride;
        lse_out[row_idx] = (l > 0.f) ? (m + lg2(l)) * 0.69314718055994531f : -INFINITY;
      }
      release_item(it);
      // The O_t reads above are complete (tcgen05.wait::ld); the PFULL
      // arrival of the next item orders them before its first P_t V.
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // Every item grab of this CTA happened before the barrier above.  The
    // last CTA to get here resets the counter pair for the next launch.
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
}

template <int D>
cudaError_t launch_persist(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const FwdParams& p, int ctas, cudaStream_t stream) {
  using C = FwdP<D>;
  auto kern = fwd_persist_kernel<D>;
  static int regs = -1;  // one per instantiation
  if (regs < 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
  }
  if (regs != kLaunchRegs) return cudaErrorInvalidKernelImage;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<ctas, kThreads, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_persist(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const FwdParams& p, int ctas, cudaStream_t stream) {
  if (d == 128) return launch_persist<128>(tmQ, tmK, tmV, p, ctas, stream);
  if (d == 64) return launch_persist<64>(tmQ, tmK, tmV, p, ctas, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
