// fwd_sm103.cu -- exact attention forward on sm_103a tensor cores.
//
// Computes O = softmax(scale * Q K^T [+ causal mask]) V and LSE per query row
// with the online (m, l, O) merge of "LLM 注意力与计算内核精读笔记 · 02
// FlashAttention" §5: per K/V tile, m+ = max(m, m~), l+ = e^{m-m+} l + rowsum(P~),
// O+ = e^{m-m+} O + P~ V.  As in FlashAttention-2 ("从Online-Softmax到
// FlashAttention V1/V2/V3", 0x05), O stays unnormalised and 1/l is applied
// once at the end; each CTA owns its query rows and loops over K/V (Q outer
// loop), so CTAs never communicate.  Causal tiles above the diagonal are never
// visited and only tiles that cross the diagonal are masked (0x09's three tile
// cases).  GQA reads K/V head h / (Hq / Hkv) by indexing (0x09).
//
// The running max may lag behind the true max: softmax(s) = e^{s-m} / sum e^{s-m}
// holds for any m (§5.1 of the same notes), so a row only moves its m (and
// rescales l and its O row) when the new tile's max exceeds it by more than
// 2^16; otherwise P~ = 2^{s - m} <= 65536, which bf16 P (8 exponent bits) and
// fp32 l, O hold with the same relative precision as values <= 1.
//
// Mapping to the hardware (one CTA = two 128-row query tiles, 12 warps):
//   warp 0      TMA producer: both Q tiles once, then K and V tiles through a
//               STAGES-deep ring of shared-memory slots (full/empty mbarriers),
//               in use order: K_0, then K_{j+1} ahead of V_j.
//   warp 1      TMEM allocator and tcgen05.mma issuer (the converged warp runs
//               the loop, one elected lane issues):
//               S_t = Q_t K_j^T  (SS MMA, M=128 N=128) into ONE shared S buffer
//               O_t += P_t V_j   (TS MMA, P_t from its own TMEM region)
//   warps 4..7  softmax of query tile 0, warps 8..11 of tile 1: thread r owns
//               row r; it loads its S row from TMEM (32x32b loads) and at once
//               releases the S buffer, so the other tile's next Q K^T runs
//               while this tile computes its exponentials; it keeps m and l in
//               registers (log2 units), writes P as packed bf16 into its own
//               64-column region once its previous P V has completed, rescales
//               its O row in TMEM when m moves, and finally writes O / l, LSE.
// The S buffer alternates S_0(j), S_1(j), S_0(j+1), ...: while one warpgroup
// computes exponentials the tensor pipe runs the other tile's P V and Q K^T.
// TMEM columns: [0,128) S, [128,192) P_0, [192,256) P_1, then O_0, O_1.
// Registers: warpgroup 0 gives registers to the two softmax warpgroups
// (setmaxnreg), which hold a whole S row each.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;  // query rows per tile (two tiles per CTA)
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;  // per-thread registers of a 384-thread CTA (3 warps per SMSP)
constexpr int kRegsLow = 72;      // warpgroup 0 after setmaxnreg.dec
constexpr int kRegsHigh = 216;    // softmax warpgroups after setmaxnreg.inc
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 16.0f;  // log2 units: rescale when m grows by > 2^16

// ONE: the one-query-tile variant holds one Q tile and gives the space to
// the K/V ring (it streams K and V for few rows: decoding).
template <int D, bool ONE = false>
struct Fwd {
  static constexpr int CB = D / 64;              // 128-byte column blocks per row
  static constexpr int BLOCK_BYTES = 128 * 128;  // one 128-row x 64-col bf16 block
  static constexpr int TILE_BYTES = CB * BLOCK_BYTES;
  static constexpr int QT = ONE ? 1 : 2;         // Q tiles held
  static constexpr int STAGES = (D == 128 ? 4 : 8) + (ONE ? 1 : 0);  // a stage = one tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = QT * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TILE_BYTES;
  static constexpr int B_QFULL = 0;
  static constexpr int B_KVFULL = 1;
  static constexpr int B_KVEMPTY = B_KVFULL + STAGES;
  static constexpr int B_SFULL = B_KVEMPTY + STAGES;  // 2: S buffer holds S_t
  static constexpr int B_SREAD = B_SFULL + 2;         // 2: S_t read out of the S buffer
  static constexpr int B_PFULL = B_SREAD + 2;         // 2
  static constexpr int B_ODONE = B_PFULL + 2;         // 2: P_t V complete
  static constexpr int B_DRAIN = B_ODONE + 2;         // 2: one per issuing warp
  static constexpr int NBARS = B_DRAIN + 2;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int OFF_NLIST = OFF_ABORT + 4;           // block-sparse: entries in the tile list
  static constexpr int OFF_LIST = OFF_NLIST + 4;            // uint16 per listed K/V tile
  static constexpr int SMEM_BYTES = OFF_LIST + 2 * kMaxMaskTiles + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB of shared memory per block");
  static constexpr uint32_t IDESC_S = idesc_bf16(kBM, kBN, false, false);
  static constexpr uint32_t IDESC_O = idesc_bf16(kBM, D, false, true);
  static constexpr uint32_t TM_S = 0;    // one S buffer shared by both tiles (128 columns)
  static constexpr uint32_t TM_P = 128;  // + 64 * t: P_t as packed bf16
  static constexpr uint32_t TM_O = 256;  // + D * t
};

// ONE: every CTA computes query tile 0 only (N <= 128: decoding and short
// sequences), with its own MMA schedule; otherwise both tiles (a last pair
// whose second tile has no row below N still computes it, on zero rows).
template <int D, bool ONE, bool MASKED>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Fwd<D, ONE>;
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
  // CTA -> (b*Hq + h, pair of query tiles), heaviest pairs first within groups of heads.
  int bh, rank;
  const int split = blockIdx.x % p.n_splits;
  grouped_order(blockIdx.x / p.n_splits, p.heads, p.n_pairs, p.head_group, bh, rank);
  const int pair = p.n_pairs - 1 - rank;
  const int q0 = pair * 2 * kBM;
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int bh_kv = p.packed ? bh : b * p.Hkv + h / (p.Hq / p.Hkv);
  // K/V tiles [kt0, kt0 + n_kv): this CTA's split of the key range, without
  // the tiles right of the causal diagonal of its last query row (never
  // loaded).  An empty range writes O = 0 and LSE = -inf.
  const int kt0 = split * p.tiles_per_split;
  int kt_end = min(kt0 + p.tiles_per_split, (p.Nk + kBN - 1) / kBN);
  if (p.causal) {
    // Last key of the tile's last query (of its largest query index when packed).
    const int k_last = (p.packed ? p.N : min(q0 + 2 * kBM, p.N)) - 1 + p.kv_off;
    kt_end = k_last < 0 ? 0 : min(kt_end, k_last / kBN + 1);
  }
  int n_kv = max(0, kt_end - kt0);
  constexpr bool two = !ONE;
  // Block-sparse: the K/V tiles of [kt0, kt_end) that either query tile keeps
  // (mask entry nonzero and not right of its causal diagonal), as a list of
  // entries kt | 0x8000 (tile 0 keeps it) | 0x4000 (tile 1 keeps it), built by
  // the otherwise idle warp 3 with a ballot compaction.
  constexpr bool masked = MASKED;  // p.bmask != NULL
  uint16_t* const tlist = reinterpret_cast<uint16_t*>(smem + C::OFF_LIST);
  int* const nlist = reinterpret_cast<int*>(smem + C::OFF_NLIST);
  if (masked && warp == 3) {
    const int nkt = (p.Nk + kBN - 1) / kBN;
    const int qa = q0 / kBM;  // the pair's first query tile
    const uint8_t* mh = p.bmask + (size_t)(p.bmask_heads == 1 ? 0 : h) * p.n_qtiles * nkt;
    int count = 0;
    for (int base = kt0; base < kt_end; base += 32) {
      const int kt = base + lane;
      uint32_t e = 0;
      if (kt < kt_end) {
        bool on0 = mh[(size_t)qa * nkt + kt] != 0;
        bool on1 = two && qa + 1 < p.n_qtiles && mh[(size_t)(qa + 1) * nkt + kt] != 0;
        if (p.causal) {
          on0 = on0 && kt * kBN <= min(q0 + kBM, p.N) - 1 + p.kv_off;
          on1 = on1 && kt * kBN <= min(q0 + 2 * kBM, p.N) - 1 + p.kv_off;
        }
        if (on0 || on1) e = (uint32_t)kt | (on0 ? 0x8000u : 0u) | (on1 ? 0x4000u : 0u);
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, e != 0);
      if (e) tlist[count + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)e;
      count += __popc(bal);
    }
    if (lane == 0) *nlist = count;
  }
  auto ktile = [&](int j) -> int { return masked ? (tlist[j] & 0x3FFF) : kt0 + j; };
  float* const o_out = p.out_f32 ? static_cast<float*>(p.O) + split * p.o_split_stride : nullptr;
  uint16_t* const o_out16 = p.out_f32 ? nullptr : static_cast<uint16_t*>(p.O);
  float* const lse_out = p.LSE + split * p.lse_split_stride;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QFULL), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::B_KVFULL + s), 1);
      mbar_init(bar(C::B_KVEMPTY + s), two ? 2 : 1);  // one commit per tile reading the slot
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_SFULL + i), 1);
      mbar_init(bar(C::B_PFULL + i), 4);  // one arrival per softmax warp
      mbar_init(bar(C::B_ODONE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_SREAD + i), 4);  // one arrival per softmax warp of tile i
      mbar_init(bar(C::B_DRAIN + i), 1);
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
  if (masked) n_kv = *nlist;
  const WaitCtx wc{abort_flag, p.status, p.wait_limit_ns};

  if (warp < 4) {
    regs_dec<kRegsLow>();
    if (warp == 0 && lane == 0 && n_kv > 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(C::B_QFULL), C::QT * C::TILE_BYTES);
      if (dcheck(q0 >= 0 && q0 < p.n_pairs * 2 * kBM && bh >= 0 && bh < p.heads, p.status))
        for (int t = 0; t < C::QT; ++t)
          for (int cb = 0; cb < C::CB; ++cb)
            tma_load_3d(sQ + t * C::TILE_BYTES + cb * C::BLOCK_BYTES, &tmQ, bar(C::B_QFULL), cb * 64,
                        q0 + t * kBM, bh);
      // Load order follows use order: K_0, then K_{j+1} before V_j (the next
      // Q K^T is issued before this tile's P V).
      int li = 0;
      bool ok = true;
      for (int u = 0; u < 2 * n_kv && ok; ++u, ++li) {
        int j;  // tile index of this load
        bool v;
        if (n_kv == 1) {
          v = (u == 1);
          j = 0;
        } else if (u == 0) {
          v = false;
          j = 0;
        } else if (u == 2 * n_kv - 1) {
          v = true;
          j = n_kv - 1;
        } else {
          v = (u % 2 == 0);
          j = v ? u / 2 - 1 : (u + 1) / 2;
        }
        const int s = li % C::STAGES;
        const uint32_t ph = (li / C::STAGES) & 1;
        if (li >= C::STAGES && !mbar_wait(bar(C::B_KVEMPTY + s), ph ^ 1, wc)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(C::B_KVFULL + s), C::TILE_BYTES);
        const CUtensorMap* m = v ? &tmV : &tmK;
        const int kt = ktile(j);
        if (dcheck(kt >= 0 && kt * kBN < p.Nk && bh_kv >= 0 && bh_kv < (p.packed ? p.heads : p.B * p.Hkv),
                   p.status))
          for (int cb = 0; cb < C::CB; ++cb)
            tma_load_3d(sKV + s * C::TILE_BYTES + cb * C::BLOCK_BYTES, m, bar(C::B_KVFULL + s), cb * 64,
                        kt * kBN, bh_kv);
      }
      // All loads are issued: a merge launched behind this kernel may start
      // (it waits for this kernel's completion before reading).
      griddep_launch_dependents();
      // Drain: every issued copy must land before the CTA may exit.
      mbar_wait_drain(bar(C::B_QFULL), 0, wc);
      for (int k = max(0, li - C::STAGES); k < li; ++k)
        mbar_wait_drain(bar(C::B_KVFULL + k % C::STAGES), (k / C::STAGES) & 1, wc);
    } else if ((warp == 1 || (two && warp == 2)) && n_kv > 0) {
      // ---------------------------------------------------------- MMA issuers
      // The whole warp runs this loop (uniform operands); one elected lane
      // issues.  Two query tiles: warp 1 issues tile 0's products and warp 2
      // tile 1's (a warp needs about as long to issue an M = N = 128 product
      // as the tensor pipe needs to run it, so two issuing warps keep the
      // pipe fed while either waits).  One tile: warp 1 alone.
      // Ring slots of the loads (see the producer): K_0 first, then K_{j+1}
      // ahead of V_j.
      const int t = warp - 1;
      auto k_li = [&](int j) -> int { return j == 0 ? 0 : 2 * j - 1; };
      auto v_li = [&](int j) -> int { return j == n_kv - 1 ? 2 * n_kv - 1 : 2 * j + 2; };
      auto kv_slot = [&](int li) -> int { return li % C::STAGES; };
      bool ok = mbar_wait_warp(bar(C::B_QFULL), 0, wc);
      auto wait_kv = [&](int li) -> bool {
        if (!mbar_wait_warp(bar(C::B_KVFULL + kv_slot(li)), (li / C::STAGES) & 1, wc)) return false;
        tc_fence_after();
        return true;
      };
      // S_t = Q_t K_j^T into the shared S buffer.
      auto issue_s = [&](int j) {
        const uint32_t kb = sKV + kv_slot(k_li(j)) * C::TILE_BYTES;
        const uint32_t qb = sQ + t * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32;
          mma_ss_warp(tmem + C::TM_S, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                      C::IDESC_S, kk > 0 ? 1u : 0u);
        }
        tc_commit_warp(bar(C::B_SFULL + t));
        tc_commit_warp(bar(C::B_KVEMPTY + kv_slot(k_li(j))));  // K_j: one commit per tile
      };
      // O_t += P_t V_j (A = 16 keys of P_t = 8 TMEM columns; B = 16 V rows, MN-major).
      auto issue_pv = [&](int j) {
        const uint32_t vb = sKV + kv_slot(v_li(j)) * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts_warp(tmem + C::TM_O + t * D, tmem + C::TM_P + t * 64 + kk * 8,
                      sdesc_sw128(vb + kk * 2048, C::BLOCK_BYTES, 1024), C::IDESC_O,
                      (kk > 0 || j > 0) ? 1u : 0u);
        tc_commit_warp(bar(C::B_ODONE + t));
        tc_commit_warp(bar(C::B_KVEMPTY + kv_slot(v_li(j))));  // V_j: one commit per tile
      };
      // The S buffer passes S_0(j), S_1(j), S_0(j+1), ... (one tile: S_0(j),
      // S_0(j+1), ...); each S is issued once the one before it has been
      // read: tile 1's S(j) after tile 0 read S_0(j), tile 0's S(j) after
      // tile 1 (one tile: tile 0) read the previous one.
      int ns = 0;  // S products of this tile issued so far
      auto wait_sbuf = [&]() -> bool {
        if (t == 0 && ns == 0) return true;
        const int other = two ? t ^ 1 : 0;
        const int phase = (t == 0) ? ns - 1 : ns;
        if (!mbar_wait_warp(bar(C::B_SREAD + other), phase & 1, wc)) return false;
        tc_fence_after();
        return true;
      };
      auto wait_p = [&](int j) -> bool {
        if (!mbar_wait_warp(bar(C::B_PFULL + t), j & 1, wc)) return false;
        tc_fence_after();
        return true;
      };
      ok = ok && wait_sbuf() && wait_kv(k_li(0));
      if (ok) {
        issue_s(0);
        ++ns;
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        if (j + 1 < n_kv) {
          if (!wait_sbuf() || !wait_kv(k_li(j + 1))) break;
          issue_s(j + 1);
          ++ns;
        }
        if (!wait_kv(v_li(j)) || !wait_p(j)) break;
        issue_pv(j);
      }
      // Drain: all MMAs of this warp complete before TMEM is released.
      tc_commit_warp(bar(C::B_DRAIN + t));
      mbar_wait_drain_warp(bar(C::B_DRAIN + t), 0, wc);
    }
  } else {
    regs_inc<kRegsHigh>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    const int quad = warp & 3;      // TMEM lane quarter this warp may access
    const int row = quad * 32 + lane;
    const int qt0 = q0 + t * kBM;
    const int q = qt0 + row;                   // row of the grid head
    const int qc = p.packed ? q % p.N : q;     // its query index (causal limit)
    const int qc0 = p.packed ? 0 : qt0;        // smallest query index in the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_t = tmem + lane_off + C::TM_S;  // shared S buffer
    const uint32_t p_t = tmem + lane_off + C::TM_P + t * 64;
    const uint32_t o_t = tmem + lane_off + C::TM_O + t * D;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running (possibly stale) max of scale*s, log2 units
    float l = 0.f;        // running sum of 2^(scale*s*log2e - m): gives LSE
    float corr = 0.f;     // sum over tiles of (largest P - its bf16 rounding), same scale as l
    bool ok = true;
    const bool active = t == 0 || two;  // tile 1 of a one-tile CTA has no rows
    for (int j = 0; j < (active ? n_kv : 0); ++j) {
      const int k0 = ktile(j) * kBN;
      const bool on = !masked || ((tlist[j] >> (15 - t)) & 1);  // this tile keeps the block
      if (!mbar_wait(bar(C::B_SFULL + t), j & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_t + c * 32, sr[c]);
      tmem_ld_wait(sr[0]);
      reg_fence32(sr[1]);
      reg_fence32(sr[2]);
      reg_fence32(sr[3]);
      // The S buffer can take the other tile's next scores now.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_SREAD + t));
      // Mask keys past N (ragged tail) and, on tiles crossing the diagonal, keys after q.
      if (!on || (k0 + kBN > p.Nk) || (p.causal && k0 + kBN - 1 > qc0 + p.kv_off)) {
        const int lim = !on ? -1 : p.causal ? min(p.Nk - 1, qc + p.kv_off) : p.Nk - 1;
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
      // Move m only when the tile's max exceeds it by more than the threshold.
      const bool move = mx > m + kRescaleThreshold;
      float alpha = 1.f;
      if (move) {
        alpha = ex2(m - mx);  // 0 when m = -inf
        m = mx;
        l *= alpha;
        corr *= alpha;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      {
        // The tile's largest P as the loop below computes it, and what its
        // rounding to bf16 (the P that multiplies V) takes away from it.
        const float pmax = ex2(fmaf(mraw, sl2, -m_use));
        corr += pmax - __uint_as_float(pack_bf16(pmax, pmax) & 0xffff0000u);
      }
      // Row sums in four packed (f32x2) accumulators; x = s * scale*log2e - m
      // for two columns per packed FMA; P kept as packed bf16 pairs.
      uint64_t rs2[4] = {0, 0, 0, 0};
      const uint64_t sl2x2 = f2pack(sl2, sl2);
      const uint64_t negm2 = f2pack(-m_use, -m_use);
      uint32_t w[2][32];
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
          w[c >> 1][(c & 1) * 16 + i] = pack_bf16(p0, p1);
        }
      {
        float a0, a1;
        f2unpack(fadd2(fadd2(rs2[0], rs2[1]), fadd2(rs2[2], rs2[3])), a0, a1);
        l += a0 + a1;
      }
      if (j > 0) {
        // P_t V of the previous tile must be complete: it reads the P_t
        // columns written below, and O_t may be rescaled.
        if (!mbar_wait(bar(C::B_ODONE + t), (j - 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, move)) {
          // The whole O row in one round trip (sr is free again).
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
      tmem_st32(p_t, w[0]);
      tmem_st32(p_t + 32, w[1]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_PFULL + t));
    }
    // Epilogue: O / l and LSE (O = 0, LSE = -inf when no key was in range).
    const bool have = n_kv > 0;
    const bool ep = ok && active && (!have || mbar_wait(bar(C::B_ODONE + t), (n_kv - 1) & 1, wc));
    // bf16 rows go out through this warp's quarter of its Q tile, free once
    // the tile's last P V -- and with it every product of the tile -- has
    // completed.  The staging needs the whole warp: a warp some of whose lanes
    // gave up (a timed-out wait, already in the status word) writes nothing.
    if (__all_sync(0xffffffffu, ep)) {
      if (have) tc_fence_after();
      // O is divided by the row sum less the rounding of each tile's largest
      // P: when one key dominates a row, its bf16 rounding then cancels
      // between O and the divisor.  LSE uses the exact sum.
      const float lo = l - corr;
      const float inv_l = lo > 0.f ? 1.f / lo : 0.f;
      const bool split_ok = dcheck(split < p.n_splits, p.status);
      const bool valid = q < p.rows && split_ok;
      const size_t row_idx = (size_t)bh * p.rows + q;
      const uint32_t sEpi = sQ + t * C::TILE_BYTES + quad * 4096;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (have) {
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
                                   __uint_as_float(o[4 * i + 2]) * inv_l,
                                   __uint_as_float(o[4 * i + 3]) * inv_l);
          } else {
            epi_stage32(sEpi, lane, c, o, inv_l);
          }
        }
        if (!p.out_f32 && (c & 1))
          epi_store_half(sEpi, lane, c >> 1, o_out16, (size_t)bh * p.rows + qt0 + quad * 32, D,
                         split_ok ? p.rows - (qt0 + quad * 32) : 0);
      }
      if (valid) {
        // LSE = ln(sum_j e^{s_j}) = (m + log2 l) * ln 2, m in log2 units.
        lse_out[row_idx] = (l > 0.f) ? (m + lg2(l)) * 0.69314718055994531f : -INFINITY;
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

template <int D, bool ONE, bool MASKED>
cudaError_t launch_one(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const FwdParams& p, cudaStream_t stream) {
  using C = Fwd<D, ONE>;
  auto kern = fwd_bf16_kernel<D, ONE, MASKED>;
  // setmaxnreg moves registers inside the launch allocation; refuse to launch
  // if the compiler gave the kernel a different per-thread count than assumed
  // (a larger split than the allocation would leave setmaxnreg.inc waiting).
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
  dim3 grid(p.heads * p.n_pairs * p.n_splits);
  kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_bf16_smem_bytes(int d) {
  return d == 128 ? Fwd<128>::SMEM_BYTES : Fwd<64>::SMEM_BYTES;
}

// Rows <= 128 (one query tile), or a block mask.  The dense two-tile case
// runs in the persistent kernel (launch_fwd_persist).
cudaError_t launch_fwd_bf16(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const FwdParams& p, cudaStream_t stream) {
  const bool one = p.rows <= kBM, m = p.bmask != nullptr;
  if (!one && !m) return cudaErrorInvalidValue;
  if (d == 128)
    return one ? (m ? launch_one<128, true, true>(tmQ, tmK, tmV, p, stream)
                    : launch_one<128, true, false>(tmQ, tmK, tmV, p, stream))
               : launch_one<128, false, true>(tmQ, tmK, tmV, p, stream);
  if (d == 64)
    return one ? (m ? launch_one<64, true, true>(tmQ, tmK, tmV, p, stream)
                    : launch_one<64, true, false>(tmQ, tmK, tmV, p, stream))
               : launch_one<64, false, true>(tmQ, tmK, tmV, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
