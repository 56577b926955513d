// fp8.cu -- FP8 (e4m3) attention forward with per-block scales, and the block
// quantizer that produces its inputs.
//
// "LLM 注意力与计算内核精读笔记 · 02 FlashAttention" §10 (FlashAttention-3 runs the
// two products on FP8 tensor cores with block quantization) and §12.2 (a scale
// per block tracks local magnitudes better than one per tensor).  Format
// readings: OCP e4m3 (largest finite 448, round to nearest even, saturating);
// a block is 128 consecutive rows of one head with scale amax / 448 (1 for an
// all-zero block) and codes e4m3(x / scale), both fp32 operations.
//
// Forward.  Query tile i (128 rows = one Q block) against key tile j (one K
// and one V block):  s = scale * sq_i * sk_j * (Qc Kc^T), the code product on
// the tensor cores (kind::f8f6f4, fp32 accumulation), the block scales folded
// into the per-tile exponent factor.  With V_j = sv_j * Vc_j and
// r_j = sv_j / max_j' sv_j' <= 1, the kernel rounds P' = P * r_j to e4m3 and
// accumulates O' += P' Vc_j, so O = max(sv) * O' / l with l summed from the
// unrounded P (fp32).  Both operands of P' Vc are K-major: V is stored
// transposed, [B, Hkv, d, Npad] with Npad = N rounded up to 16.
//
// Running max: as the bf16 forward, m lags the true max by up to 2^4, and the
// exponent is offset by +4, so P' <= 2^8 < 448 and the rounding of small
// probabilities is 2^4 finer than with max P = 1.  O is divided by l less the
// rounding of each tile's largest P' (cancels it when one key dominates).
//
// Mapping (one CTA = two 128-row query tiles, 12 warps): warp 0 TMA producer
// (Q tiles once, then K_j and Vt_j through an 8-slot ring), warp 1 TMEM
// allocator and MMA issuer of tile 0, warp 2 MMA issuer of tile 1 (S_t = Q_t
// K_j^T into one shared S buffer, O_t += P'_t Vt_j^T with P'_t in shared
// memory), warps 4..7 / 8..11 softmax of tile 0 / 1, one row per thread.
// TMEM: [0,128) S, [128,256) O_0, [256,384) O_1.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

// ------------------------------------------------------------------ quantizer
constexpr int kQBlock = 128;  // rows per scale block
constexpr float kE4m3Max = 448.f;

// One CTA per (head, 128-row block): amax, scale, codes.  X bf16 [BH, N, D].
// Row-major codes [BH, N, D]; transposed codes [BH, D, ldt] (columns >= N zero).
template <int D>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const uint16_t* __restrict__ X,
                                                           uint8_t* __restrict__ codes,
                                                           float* __restrict__ scales, int N, int T,
                                                           int transpose, int ldt) {
  constexpr int CH = D / 8;                  // 16-byte chunks (8 bf16) per row
  constexpr int PER = kQBlock * CH / 256;    // chunks per thread
  constexpr int TSTRIDE = kQBlock + 4;       // bytes per row of the transpose buffer
  __shared__ float red[8];
  __shared__ __align__(16) uint8_t tb[D * TSTRIDE];
  const int t = blockIdx.x % T;
  const long long bh = blockIdx.x / T;
  const int r0 = t * kQBlock;
  const int rows = min(kQBlock, N - r0);
  const uint16_t* src = X + ((size_t)bh * N + r0) * D;
  uint4 v[PER];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int u = threadIdx.x + i * 256;
    const int r = u / CH, c = u % CH;
    v[i] = r < rows ? __ldg(reinterpret_cast<const uint4*>(src + (size_t)r * D + c * 8)) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xffff0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) amax = fmaxf(amax, red[k]);
  const float sc = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
  if (threadIdx.x == 0) scales[bh * T + t] = sc;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int u = threadIdx.x + i * 256;
    const int r = u / CH, c = u % CH;
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    float x[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __fdiv_rn(__uint_as_float(w[k] << 16), sc);
      x[2 * k + 1] = __fdiv_rn(__uint_as_float(w[k] & 0xffff0000u), sc);
    }
    const uint32_t lo = pack_e4m3x4(x[0], x[1], x[2], x[3]);
    const uint32_t hi = pack_e4m3x4(x[4], x[5], x[6], x[7]);
    if (!transpose) {
      if (r < rows)
        *reinterpret_cast<uint2*>(codes + ((size_t)bh * N + r0 + r) * D + c * 8) = make_uint2(lo, hi);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tb[(c * 8 + k) * TSTRIDE + r] = (uint8_t)(lo >> (8 * k));
        tb[(c * 8 + 4 + k) * TSTRIDE + r] = (uint8_t)(hi >> (8 * k));
      }
    }
  }
  if (transpose) {
    __syncthreads();
    // Row c of the block: keys [r0, r0 + cols) of column c, in 16-byte pieces.
    const int cols = min(kQBlock, ldt - r0);  // a multiple of 16
    for (int u = threadIdx.x; u < D * 8; u += 256) {
      const int c = u >> 3, k = u & 7;
      if (16 * k >= cols) continue;
      const uint32_t* s = reinterpret_cast<const uint32_t*>(tb + c * TSTRIDE + 16 * k);
      *reinterpret_cast<uint4*>(codes + ((size_t)bh * D + c) * ldt + r0 + 16 * k) = make_uint4(s[0], s[1], s[2], s[3]);
    }
  }
}

// ------------------------------------------------------------------ forward
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 72;
constexpr int kRegsHigh = 216;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr float kThreshold = 4.0f;  // log2 units: m moves when the tile max exceeds it by > 2^4
constexpr float kShift = 4.0f;      // exponent offset: P' <= 2^(4 + 4) = 256

struct F8 {
  static constexpr int TILE = kBM * 128;  // one 128 x 128 e4m3 tile (8-row swizzle atoms)
  static constexpr int STAGES = 8;
  static constexpr int OFF_Q = 0;         // two Q tiles
  static constexpr int OFF_P = 2 * TILE;  // two P' tiles
  static constexpr int OFF_KV = 4 * TILE;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TILE;
  static constexpr int B_QFULL = 0;
  static constexpr int B_KVFULL = 1;
  static constexpr int B_KVEMPTY = B_KVFULL + STAGES;
  static constexpr int B_SFULL = B_KVEMPTY + STAGES;  // 2
  static constexpr int B_SREAD = B_SFULL + 2;         // 2: S_t read out of the S buffer
  static constexpr int B_PFULL = B_SREAD + 2;         // 2
  static constexpr int B_ODONE = B_PFULL + 2;         // 2
  static constexpr int B_DRAIN = B_ODONE + 2;         // 2: one per issuing warp
  static constexpr int NBARS = B_DRAIN + 2;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;
  static constexpr uint32_t IDESC = idesc_e4m3(kBM, kBN);  // S (N = keys) and O (N = d = 128)
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 128;  // + 128 * t
};
static_assert(F8::SMEM_BYTES <= 232448, "shared memory");

__global__ void __launch_bounds__(kThreads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmVt, const Fp8FwdParams p) {
  using C = F8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q;
  const uint32_t sP = sb + C::OFF_P;
  const uint32_t sKV = sb + C::OFF_KV;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int bh, rank;
  grouped_order(blockIdx.x, p.heads, p.n_pairs, p.head_group, bh, rank);
  const int pair = p.n_pairs - 1 - rank;
  const int q0 = pair * 2 * kBM;
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int bh_kv = b * p.Hkv + h / (p.Hq / p.Hkv);
  int n_kv = p.T;  // key tiles visited: all, or up to the causal diagonal of the last row
  if (p.causal) n_kv = min(n_kv, (min(q0 + 2 * kBM, p.N) - 1) / kBN + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QFULL), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::B_KVFULL + s), 1);
      mbar_init(bar(C::B_KVEMPTY + s), 2);  // a K or V tile is read by both tiles' products
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_SFULL + i), 1);
      mbar_init(bar(C::B_PFULL + i), 4);
      mbar_init(bar(C::B_ODONE + i), 1);
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

  if (warp < 4) {
    regs_dec<kRegsLow>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmVt);
      mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::TILE);
      for (int t = 0; t < 2; ++t) tma_load_3d(sQ + t * C::TILE, &tmQ, bar(C::B_QFULL), 0, q0 + t * kBM, bh);
      // Use order: K_0, then K_{j+1} ahead of V_j.
      int li = 0;
      for (int u = 0; u < 2 * n_kv; ++u, ++li) {
        int j;
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
        if (li >= C::STAGES && !mbar_wait(bar(C::B_KVEMPTY + s), ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(bar(C::B_KVFULL + s), C::TILE);
        if (v)
          tma_load_3d(sKV + s * C::TILE, &tmVt, bar(C::B_KVFULL + s), j * kBN, 0, bh_kv);
        else
          tma_load_3d(sKV + s * C::TILE, &tmK, bar(C::B_KVFULL + s), 0, j * kBN, bh_kv);
      }
      mbar_wait_drain(bar(C::B_QFULL), 0, wc);
      for (int k = max(0, li - C::STAGES); k < li; ++k)
        mbar_wait_drain(bar(C::B_KVFULL + k % C::STAGES), (k / C::STAGES) & 1, wc);
    } else if (warp == 1 || warp == 2) {
      // ---------------------------------------------------------- MMA issuers
      // Warp 1 issues query tile 0's products, warp 2 tile 1's (a warp needs
      // about as long to issue one of these products as the tensor pipe
      // needs to run it; two issuing warps keep the pipe fed while either
      // waits).  Per tile: S_t(0), then S_t(j+1) ahead of P'_t(j) Vt_j.  The
      // one S buffer alternates S_0(j), S_1(j), S_0(j+1): tile 1's S(j)
      // waits until tile 0 has read S_0(j), tile 0's S(j+1) until tile 1 has
      // read S_1(j).
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
      int ns = 0;  // S products of this tile issued so far
      auto wait_sbuf = [&]() -> bool {
        if (t == 0 && ns == 0) return true;
        const int phase = t == 0 ? ns - 1 : ns;
        if (!mbar_wait_warp(bar(C::B_SREAD + (t ^ 1)), phase & 1, wc)) return false;
        tc_fence_after();
        return true;
      };
      // S_t = Q_t K_j^T: four K = 32 steps along the 128-byte rows.
      auto issue_s = [&](int j) {
        const uint32_t kb = sKV + kv_slot(k_li(j)) * C::TILE;
        const uint32_t qb = sQ + t * C::TILE;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss_f8_warp(tmem + C::TM_S, sdesc_sw128(qb + kk * 32, 16, 1024),
                         sdesc_sw128(kb + kk * 32, 16, 1024), C::IDESC, kk > 0 ? 1u : 0u);
        tc_commit_warp(bar(C::B_SFULL + t));
        tc_commit_warp(bar(C::B_KVEMPTY + kv_slot(k_li(j))));  // one of K_j's two readers
        ++ns;
      };
      // O_t += P'_t Vt_j^T: A = P'_t [query rows x keys], B = Vt_j [d rows x keys].
      auto issue_pv = [&](int j) {
        const uint32_t vb = sKV + kv_slot(v_li(j)) * C::TILE;
        const uint32_t pb = sP + t * C::TILE;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss_f8_warp(tmem + C::TM_O + t * 128, sdesc_sw128(pb + kk * 32, 16, 1024),
                         sdesc_sw128(vb + kk * 32, 16, 1024), C::IDESC, (kk > 0 || j > 0) ? 1u : 0u);
        tc_commit_warp(bar(C::B_ODONE + t));
        tc_commit_warp(bar(C::B_KVEMPTY + kv_slot(v_li(j))));  // one of V_j's two readers
      };
      if (ok) ok = wait_sbuf() && wait_kv(k_li(0));
      if (ok) issue_s(0);
      for (int j = 0; j < n_kv && ok; ++j) {
        if (j + 1 < n_kv) {
          if (!wait_sbuf() || !wait_kv(k_li(j + 1))) break;
          issue_s(j + 1);
        }
        if (!wait_kv(v_li(j)) || !mbar_wait_warp(bar(C::B_PFULL + t), j & 1, wc)) break;
        tc_fence_after();
        issue_pv(j);
      }
      tc_commit_warp(bar(C::B_DRAIN + t));
      mbar_wait_drain_warp(bar(C::B_DRAIN + t), 0, wc);
    }
  } else {
    regs_inc<kRegsHigh>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int qt0 = q0 + t * kBM;
    const int q = qt0 + row;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_t = tmem + lane_off + C::TM_S;
    const uint32_t o_t = tmem + lane_off + C::TM_O + t * 128;
    const uint32_t p_row = sP + t * C::TILE + row * 128;  // this row of P'_t (128 bytes, swizzled)
    const uint32_t swz = row & 7;
    const float* skh = p.sk + (size_t)bh_kv * p.T;
    const float* svh = p.sv + (size_t)bh_kv * p.T;
    // Exponent factor of the query block, and the largest V scale this CTA uses.
    const float fq = p.scale_log2 * (qt0 < p.N ? p.sq[(size_t)bh * p.T + qt0 / kBM] : 1.f);
    float svm = 0.f;
    for (int k = lane; k < n_kv; k += 32) svm = fmaxf(svm, svh[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, o));
    const float lsvm = lg2(svm);
    float m = -INFINITY;  // running (possibly stale) max of the scaled score, log2 units
    float l = 0.f;        // sum of 2^(s*log2e - m + shift) over the keys seen
    float corr = 0.f;     // sum over tiles of (largest P' - its e4m3 rounding) / r_j
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int k0 = j * kBN;
      const float skj = skh[j];
      const float svj = svh[j];
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_SREAD + t));
      if (k0 + kBN > p.N || (p.causal && k0 + kBN - 1 > qt0)) {
        const int lim = p.causal ? min(p.N - 1, q) : p.N - 1;
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
      const float f = fq * skj;  // > 0: scale * sq * sk * log2(e)
      const float mx = mraw * f;
      const bool move = mx > m + kThreshold;
      float alpha = 1.f;
      if (move) {
        alpha = ex2(m - mx);
        m = mx;
        l *= alpha;
        corr *= alpha;
      }
      // x = S f - (m - shift) + log2 r_j, so P' = 2^x = P r_j.
      const float m_use = (m == -INFINITY) ? 0.f : m - kShift;
      const float lr = lg2(svj) - lsvm;
      const float rinv = ex2(-lr);
      const float bias = lr - m_use;
      {
        const float pmax = ex2(fmaf(mraw, f, bias));
        corr += rinv * (pmax - round_e4m3(pmax));
      }
      uint64_t rs2[4] = {0, 0, 0, 0};
      const uint64_t f2 = f2pack(f, f);
      const uint64_t b2 = f2pack(bias, bias);
      uint32_t w[32];  // P' of the row as e4m3, keys 4k..4k+3 in word k
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float x0, x1, x2, x3;
          f2unpack(ffma2(f2pack(__uint_as_float(sr[c][4 * i]), __uint_as_float(sr[c][4 * i + 1])), f2, b2), x0, x1);
          f2unpack(ffma2(f2pack(__uint_as_float(sr[c][4 * i + 2]), __uint_as_float(sr[c][4 * i + 3])), f2, b2), x2,
                   x3);
          const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
          rs2[i & 3] = fadd2(rs2[i & 3], fadd2(f2pack(p0, p1), f2pack(p2, p3)));
          w[c * 8 + i] = pack_e4m3x4(p0, p1, p2, p3);
        }
      {
        float a0, a1;
        f2unpack(fadd2(fadd2(rs2[0], rs2[1]), fadd2(rs2[2], rs2[3])), a0, a1);
        l += rinv * (a0 + a1);
      }
      if (j > 0) {
        // P'_t V of the previous tile must be complete: it reads the P'_t
        // tile written below, and O_t may be rescaled.
        if (!mbar_wait(bar(C::B_ODONE + t), (j - 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, move)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(o_t + c * 32, sr[c]);
          tmem_ld_wait(sr[0]);
#pragma unroll
          for (int c = 1; c < 4; ++c) reg_fence32(sr[c]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int i = 0; i < 32; ++i) sr[c][i] = __float_as_uint(__uint_as_float(sr[c][i]) * alpha);
            tmem_st32(o_t + c * 32, sr[c]);
          }
          tmem_st_wait();
        }
      }
      // Row of P'_t in the 128-byte-swizzled K-major layout the MMA reads:
      // 16-byte chunk c (keys 16c..16c+15) at chunk position c ^ (row & 7).
#pragma unroll
      for (int c = 0; c < 8; ++c)
        sts_u4(p_row + ((c ^ swz) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_PFULL + t));
    }
    // Epilogue: O = max(sv) O' / (l - corr), LSE = (m - shift + log2 l) ln 2.
    // bf16 rows go out through this warp's quarter of the tile's P' buffer,
    // free once the tile's last P' V has completed.  The staging needs the
    // whole warp: a warp some of whose lanes gave up (a timed-out wait, already
    // in the status word) writes nothing.
    const bool ep = ok && mbar_wait(bar(C::B_ODONE + t), (n_kv - 1) & 1, wc);
    if (__all_sync(0xffffffffu, ep)) {
      tc_fence_after();
      const float lo = l - corr;
      const float inv_l = lo > 0.f ? svm / lo : 0.f;
      const bool valid = q < p.N;
      const size_t row_idx = (size_t)bh * p.N + q;
      const uint32_t sEpi = sP + t * C::TILE + quad * 4096;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(o_t + c * 32, o);
        tmem_ld_wait(o);
        if (valid) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + row_idx * 128 + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                   __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
          } else {
            epi_stage32(sEpi, lane, c, o, inv_l);
          }
        }
        if (!p.out_f32 && (c & 1))
          epi_store_half(sEpi, lane, c >> 1, static_cast<uint16_t*>(p.O), (size_t)bh * p.N + qt0 + quad * 32, 128,
                         p.N - (qt0 + quad * 32));
      }
      if (valid) p.LSE[row_idx] = (l > 0.f) ? (m - kShift + lg2(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(int d, const uint16_t* X, uint8_t* codes, float* scales, long long BH, int N,
                                int transpose, int ldt, cudaStream_t stream) {
  const int T = (N + kQBlock - 1) / kQBlock;
  const long long blocks = BH * T;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (d == 128)
    quantize_fp8_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(X, codes, scales, N, T, transpose, ldt);
  else if (d == 64)
    quantize_fp8_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(X, codes, scales, N, T, transpose, ldt);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmVt,
                           const Fp8FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_fp8_kernel;
  static int regs = -1;
  if (regs < 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
  }
  // setmaxnreg moves registers inside the launch allocation: refuse to launch
  // with a per-thread count other than the one the split was sized for.
  if (regs != kLaunchRegs) return cudaErrorInvalidKernelImage;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F8::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<p.heads * p.n_pairs, kThreads, F8::SMEM_BYTES, stream>>>(tmQ, tmK, tmVt, p);
  return cudaGetLastError();
}

}  // namespace attn
