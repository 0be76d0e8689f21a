// fa_fwd_d128.cu — FlashAttention forward for fp16 / bf16 with head dimension 128 on sm_103a.
//
// Algorithm: the tiled online-softmax recurrence of the MUSA SDK guide
// ("FlashAttention 优化", "FlashAttention 完整算法", formula steps 1-4 and the
// flow chart): a Q tile stays resident, K/V tiles stream past it, for each
// tile S = Q K^T, the running row max m and denominator l are updated, O is
// rescaled by exp(m_old - m_new) before the new P V is added (the dataflow
// page, section 2.3, stresses that order), and O is divided by l at the end.
// The loop order (Q outer, K/V inner, Q loaded once) is the dataflow page's
// section 2.2; the parallelisation over Q blocks is the guide's
// FlashAttention-2 "sequence parallelism" note; keeping the tensor core busy
// with the next tile's Q K^T while the softmax of the current tile runs is the
// guide's FlashAttention-3 note on overlapping softmax with the GEMMs.
//
// GB300 mapping (one CTA per (batch*head, 256-row Q block, key range), 12 warps):
//   warp 9      TMA producer: Q0/Q1 once, then K_j and V_j (64 keys x 128) into
//               a 4-stage K ring and a 6-stage V ring
//   warps 8, 10 MMA warps, one per Q sub-tile i (one elected lane issues;
//               warp 8 also owns TMEM): S_i(j) = Q_i K_j^T (SS, 128 x 64 x 128)
//               into S buffer j % 2 of sub-tile i; O_i += P_i(j) V_j (TS,
//               128 x 128 x 64: P from TMEM, V MN-major). S_i(j+2) is issued
//               right behind P_i(j) V_j, whose P it overwrites (one CTA's MMAs
//               execute in issue order; -DFA_STRICT_MMA_ORDER waits for the
//               P V to complete instead), so while the softmax works on tile j
//               the tensor core computes S_i(j+1): each sub-tile's softmax
//               runs tile after tile without waiting for its own products
//   warps 0-3   softmax for Q rows 0-127   (thread = row; TMEM lanes = rows)
//   warps 4-7   softmax for Q rows 128-255
//   warp 11     idle (completes the third warpgroup)
// TMEM (512 columns): S buffers [0,64) [64,128) (sub-tile 0), [128,192)
// [192,256) (sub-tile 1), O0 [256,384), O1 [384,512). P_i(j) (16-bit, packed
// in pairs) overwrites the first 32 columns of its S buffer.
// Stage releases are mbarrier arrivals of the softmax warps, not commits in
// the MMA issue stream: S_i(j) complete means K_j has been read, and (issued
// after P_i(j-2) V_{j-2} by the same warp) that V_{j-2} has been read too.
// The rescale of O is lazy and optimistic: P is computed against the current
// reference max without a max over the tile, and the max is taken (the
// reference moved, l and O rescaled, P recomputed) only when a row's P sum
// exceeds 2^15 (so P <= 2^15); a rescale at tile j needs P_i(j-1) V
// complete, which the completion of S_i(j+1) (issued after it) shows, or for
// the last tile a commit made after P_i(nkv-2) V.
// The epilogue divides by l, rounds to the input type, stages the tile in the
// sub-tile's (no longer read) Q buffer in the TMA 128-byte swizzle layout and
// TMA-stores it; LSE = ln2 * (m + log2 l) is written per row.
#include <atomic>

#include "fa_device_common.cuh"

namespace fa {
namespace {

constexpr float kLog2e128 = 1.4426950408889634f;
constexpr float kLn2_128 = 0.6931471805599453f;

struct C128 {
  static constexpr int D = 128;
  static constexpr int BM = kF16BlockQ;    // Q rows per sub-tile (= TMEM lanes)
  static constexpr int BN = kD128BlockKV;  // keys per K/V tile
  static constexpr int KST = 4;            // K ring stages
  static constexpr int VST = 6;            // V ring stages (a V stage is held two tiles longer than a K stage)
  static constexpr uint32_t ROW = 128;                // one 128-byte swizzle row = 64 elements
  static constexpr uint32_t Q_SUB = BM * D * 2;       // one Q sub-tile (32 KB)
  static constexpr uint32_t Q_HALF = BM * ROW;        // 64 columns of a Q sub-tile (16 KB)
  static constexpr uint32_t KV_BYTES = BN * D * 2;    // one K or V tile (16 KB)
  static constexpr uint32_t KV_HALF = BN * ROW;       // 64 columns of a K or V tile (8 KB)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * Q_SUB;
  static constexpr uint32_t OFF_V = OFF_K + KST * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + VST * KV_BYTES;
  // barriers: q | k_full[KST] | k_empty[KST] | v_full[VST] | v_empty[VST] |
  //           s_full[sub][buf] | p_full[sub][buf] | o_prev_last[sub] | o_last[sub] |
  //           pv_done[sub] (strict build) | drain[sub]
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1, B_KE = B_KF + KST, B_VF = B_KE + KST, B_VE = B_VF + VST;
  static constexpr int B_SF = B_VE + VST, B_PF = B_SF + 4, B_OP = B_PF + 4, B_OL = B_OP + 2, B_PVD = B_OL + 2;
  static constexpr int B_DRAIN = B_PVD + 2;
  static constexpr int NBAR = B_DRAIN + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;       // [0] TMEM base, [1] abort flag
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_O0 = 256, T_O1 = 384;
  static constexpr int THREADS = 384;
  static constexpr int WARP_MMA0 = 8, WARP_TMA = 9, WARP_MMA1 = 10;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(4 * BN + 2 * D == TMEM_COLS, "TMEM layout: four S buffers and two O accumulators");
  // Under the causal mask sub-tile 1 runs two tiles past sub-tile 0 (its 128
  // extra rows see 128 more keys), and sub-tile 0 never frees the stages of
  // what it does not read: its last K release is for K_{nkv0-1}, its last V
  // release for V_{nkv0-3}, while the producer loads up to tile nkv0+1. The
  // rings must be deep enough that those loads wait on no later release.
  static_assert(KST >= 2 && VST >= 4, "ring depth needed by unequal sub-tile tile counts");
};

__device__ __forceinline__ uint32_t bar128(uint32_t base, int i) { return base + C128::OFF_BAR + 8u * i; }

// TMEM column of S buffer `buf` of sub-tile `sub` (P overwrites its first 32 columns).
__device__ __forceinline__ uint32_t t_s128(int sub, int buf) { return 64u * (2 * sub + buf); }

// A descriptor the compiler must treat as computed here, so that unrolled
// k-loops do not make it hoist every k-step's descriptor into registers.
__device__ __forceinline__ uint64_t opaque128(uint64_t x) {
  asm volatile("" : "+l"(x));
  return x;
}

// --------------------------------------------------------------------------
// TMA producer (one thread)
// --------------------------------------------------------------------------
__device__ __forceinline__ void producer128(const FwdParams& p, uint32_t base, int bh, int row0, int nkv0, int nkv1,
                                            int t0, const WaitCtl& ctl) {
  using C = C128;
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);
  tma_prefetch_desc(&p.tm_o);
  // Q of a sub-tile with no key tile (key length 0, or a key range past its
  // rows under the causal mask) is not loaded: its epilogue may write into
  // that Q buffer, where no copy may land. A unit with no key tile at all
  // loads nothing.
  const int nkv = max(nkv0, nkv1);
  if (nkv == 0) return;
  const uint32_t bq = bar128(base, C::B_Q);
  mbar_arrive_expect_tx(bq, ((nkv0 > 0 ? 1u : 0u) + (nkv1 > 0 ? 1u : 0u)) * C::Q_SUB);
  for (int sub = 0; sub < 2; ++sub) {
    if ((sub ? nkv1 : nkv0) == 0) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      tma_load_3d(base + C::OFF_Q + sub * C::Q_SUB + h * C::Q_HALF, &p.tm_q, bq, 64 * h, row0 + C::BM * sub, bh);
  }

  int nk = 0, nv = 0;  // K / V tiles whose loads were issued
  for (int j = 0; j < nkv; ++j) {
    const int ks = j % C::KST, vs = j % C::VST;
    if (!wait_bar(bar128(base, C::B_KE + ks), ((j / C::KST) & 1) ^ 1, ctl, kWhereKEmpty)) break;
    const uint32_t kf = bar128(base, C::B_KF + ks);
    mbar_arrive_expect_tx(kf, C::KV_BYTES);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      tma_load_3d(base + C::OFF_K + ks * C::KV_BYTES + h * C::KV_HALF, &p.tm_k, kf, 64 * h, (t0 + j) * C::BN, bh);
    nk = j + 1;
    FA_TRACE(p, kEvKIssued, j);
#ifdef FA_TESTING
    if (p.inject == 1 && j == 0) continue;  // fault injection: V_0 is never loaded
#endif
    if (!wait_bar(bar128(base, C::B_VE + vs), ((j / C::VST) & 1) ^ 1, ctl, kWhereVEmpty)) break;
    const uint32_t vf = bar128(base, C::B_VF + vs);
    mbar_arrive_expect_tx(vf, C::KV_BYTES);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      tma_load_3d(base + C::OFF_V + vs * C::KV_BYTES + h * C::KV_HALF, &p.tm_v, vf, 64 * h, (t0 + j) * C::BN, bh);
    nv = j + 1;
    FA_TRACE(p, kEvVIssued, j);
  }
  // Drain, always (the loop ended, this thread's wait gave up, or another role
  // may abort later): every copy this thread started must land before the CTA
  // exits. The most recent load of each stage is one of the last KST (VST)
  // tiles issued. Cheap when nothing failed: the consumers need these copies.
  wait_bar_drain(bq, 0, ctl);
  for (int t = nk > C::KST ? nk - C::KST : 0; t < nk; ++t)
    wait_bar_drain(bar128(base, C::B_KF + t % C::KST), (t / C::KST) & 1, ctl);
  for (int t = nv > C::VST ? nv - C::VST : 0; t < nv; ++t) {
#ifdef FA_TESTING
    if (p.inject == 1 && t == 0) continue;  // never armed
#endif
    wait_bar_drain(bar128(base, C::B_VF + t % C::VST), (t / C::VST) & 1, ctl);
  }
}

// --------------------------------------------------------------------------
// MMA warp of Q sub-tile SUB (whole warp; one elected lane issues)
// --------------------------------------------------------------------------
template <bool BF16, int SUB>
__device__ __forceinline__ void mma128(const FwdParams& p, uint32_t base, uint32_t tmem, int nkv, const WaitCtl& ctl) {
  using C = C128;
  constexpr uint32_t fmt = BF16 ? 1u : 0u;
  // S = Q K^T: A = Q (K-major), B = K tile (K-major), M = 128, N = 64.
  constexpr uint32_t idesc_qk = make_idesc(fmt, 0, 0, 128, C::BN);
  // O += P V: A = P from TMEM (K-major), B = V tile, N (= d) contiguous -> MN-major.
  constexpr uint32_t idesc_pv = make_idesc(fmt, 0, 1, 128, C::D);
  const uint32_t qbase = base + C::OFF_Q + SUB * C::Q_SUB;
  const uint32_t d_o = tmem + (SUB ? C::T_O1 : C::T_O0);
  const uint32_t b_drain = bar128(base, C::B_DRAIN + SUB);
  (void)p;

  // S_i(j) = Q_i K_j^T into S buffer j % 2 (8 k-steps of 16 over d = 128; the
  // 16 elements of a k-step are 32 bytes inside the swizzled row, and every 4
  // k-steps move to the next 64-column half).
  auto issue_s = [&](int j) {
    const uint64_t a0 = opaque128(smem_desc_sw128(qbase, 16, 1024));
    const uint64_t b0 = opaque128(smem_desc_sw128(base + C::OFF_K + (j % C::KST) * C::KV_BYTES, 16, 1024));
#pragma unroll
    for (int kk = 0; kk < C::D / 16; ++kk) {
      const uint32_t aoff = ((kk / 4) * C::Q_HALF + (kk & 3) * 32u) >> 4;
      const uint32_t boff = ((kk / 4) * C::KV_HALF + (kk & 3) * 32u) >> 4;
      mma_f16_ss_elect(tmem + t_s128(SUB, j & 1), a0 + aoff, b0 + boff, idesc_qk, kk > 0 ? 1u : 0u);
    }
    tc_commit_elect(bar128(base, C::B_SF + 2 * SUB + (j & 1)));
    FA_TRACE(p, kEvS0Issued + SUB, j);
  };

  if (nkv == 0) goto drain;  // no key to attend to (key length 0): nothing to issue
  if (!wait_bar_warp(bar128(base, C::B_Q), 0, ctl, kWhereQ)) goto drain;
  for (int j = 0; j < nkv && j < 2; ++j) {
    if (!wait_bar_warp(bar128(base, C::B_KF + j % C::KST), (j / C::KST) & 1, ctl, kWhereKFull)) goto drain;
    tc_fence_after();
    issue_s(j);
  }
  for (int j = 0; j < nkv; ++j) {
    // O_i += P_i(j) V_j: 4 k-steps of 16 keys (two 8-row swizzle atoms, SBO
    // apart); the two 64-wide halves of d are LBO = 8 KB apart.
    const int vs = j % C::VST;
    if (!wait_bar_warp(bar128(base, C::B_VF + vs), (j / C::VST) & 1, ctl, kWhereVFull)) goto drain;
    if (!wait_bar_warp(bar128(base, C::B_PF + 2 * SUB + (j & 1)), (j >> 1) & 1, ctl, kWherePFull)) goto drain;
    tc_fence_after();
    if (SUB == 0) FA_TRACE(p, kEvMmaVFull, j);
    {
      const uint64_t v0 = opaque128(smem_desc_sw128(base + C::OFF_V + vs * C::KV_BYTES, C::KV_HALF, 1024));
      const uint32_t a_p = tmem + t_s128(SUB, j & 1);
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_f16_ts_elect(d_o, a_p + kk * 8, v0 + ((kk * 16 * C::ROW) >> 4), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
    }
#ifdef FA_STRICT_MMA_ORDER
    tc_commit_elect(bar128(base, C::B_PVD + SUB));
#endif
    if (j == nkv - 2) tc_commit_elect(bar128(base, C::B_OP + SUB));  // a rescale at the last tile waits for it
    if (j == nkv - 1) tc_commit_elect(bar128(base, C::B_OL + SUB));  // the epilogue waits for it
    FA_TRACE(p, kEvPV0Issued + SUB, j);
    if (j + 2 < nkv) {
      // S_i(j+2) into the columns of P_i(j), right behind the P_i(j) V_j that
      // reads them (the strict build waits for that P V to complete first).
#ifdef FA_STRICT_MMA_ORDER
      if (!wait_bar_warp(bar128(base, C::B_PVD + SUB), j & 1, ctl, kWhereODone)) goto drain;
#endif
      const int n = j + 2;
      if (!wait_bar_warp(bar128(base, C::B_KF + n % C::KST), (n / C::KST) & 1, ctl, kWhereKFull)) goto drain;
      tc_fence_after();
      if (SUB == 0) FA_TRACE(p, kEvMmaKFull, n);
      issue_s(n);
    }
  }
drain:
  // All MMAs issued by this warp complete before the CTA may free TMEM / exit.
  tc_commit_elect(b_drain);
  __all_sync(0xffffffffu, wait_bar_drain(b_drain, 0, ctl));
}

// --------------------------------------------------------------------------
// Softmax + lazy correction + epilogue (one warpgroup per Q sub-tile)
// --------------------------------------------------------------------------
template <bool BF16>
__device__ __forceinline__ void softmax128(const FwdParams& p, uint32_t base, uint32_t tmem, int sub, int bh, int row0,
                                           int split, int t0, int nkv, int key_end, const WaitCtl& ctl) {
  using C = C128;
  const int t = threadIdx.x - sub * 128;  // row within the sub-tile
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = static_cast<uint32_t>(t & ~31) << 16;
  const uint32_t t_o = tmem + lane_base + (sub ? C::T_O1 : C::T_O0);
  const float c = p.scale * kLog2e128;  // scores in log2 units: x = s * c
  // Keys this row may see: [0, row_end) (all keys up to key_end; causal: up to the row itself).
  const int my_row = row0 + C::BM * sub + t;
  const int row_end = p.causal ? min(key_end, my_row + 1) : key_end;
  // Largest sum of a tile's P, against the reference max, that leaves the
  // reference where it is: 2^tau.
  const float p_limit = ex2_approx(rescale_threshold(p));

  float m_ref = -INFINITY;  // reference max (log2 units) shared by l and O
  float l = 0.f;            // sum of P (fp32) relative to m_ref: gives LSE
  float l_o = 0.f;          // bf16 only: sum of the rounded P: normalises O
  bool ok = true;
  bool s_waited = false;    // S of this tile already waited for (by the previous tile's rescale)

  for (int j = 0; j < nkv; ++j) {
    const int b = j & 1;
    const uint32_t t_s = tmem + lane_base + t_s128(sub, b);
    // Wait results are made warp-uniform: TMEM loads/stores below need the whole warp.
    if (!s_waited && !__all_sync(0xffffffffu, wait_bar(bar128(base, C::B_SF + 2 * sub + b), (j >> 1) & 1, ctl,
                                                         kWhereSFull))) {
      ok = false;
      break;
    }
    s_waited = false;
    tc_fence_after();
    if (t == 0) FA_TRACE(p, kEvSm0SFull + 2 * sub, j);
    if (lane == 0) {
      // S(j) is complete: K_j has been read, and so has V_{j-2} (P(j-2) V was
      // issued before S(j) by the same warp, and the commit covers it). V
      // first: once the producer sees a K phase complete, every warp's earlier
      // V arrival has happened.
      if (j >= 2) mbar_arrive(bar128(base, C::B_VE + (j - 2) % C::VST));
      mbar_arrive(bar128(base, C::B_KE + j % C::KST));
    }
    uint32_t sraw[2][32];
    tmem_ld32(t_s, sraw[0]);
    tmem_ld32(t_s + 32, sraw[1]);
    tmem_ld_wait();
    reg_fence(sraw[0]);
    reg_fence(sraw[1]);
    if (t == 0) FA_TRACE(p, kEvSm0Loaded + 4 * sub, j);
    float s[C::BN];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      s[u] = __uint_as_float(sraw[0][u]);
      s[32 + u] = __uint_as_float(sraw[1][u]);
    }
    const int valid = row_end - (t0 + j) * C::BN;  // keys of this tile this row may see
    if (valid < C::BN) {
#pragma unroll
      for (int u = 0; u < C::BN; ++u)
        if (u >= valid) s[u] = -INFINITY;
    }
    // P = 2^(s*c - m_ref), two scores per packed FMA, stored over the S
    // columns as packed 16-bit pairs. The exact fp32 sum gives l (for LSE);
    // for bf16 the P.V product sees P rounded to 8 significant bits, so O is
    // normalised by the sum of the rounded P (l_o): numerator and denominator
    // then use the same weights.
    //
    // The reference max is lazy and optimistic: P is first computed against
    // the current m_ref, with no max over the tile (the max and the vote on
    // it would hold every exponential of the tile behind a reduction over all
    // its scores). Only when a row's P sum exceeds 2^tau (any row of the warp:
    // TMEM access is per warp) is the tile's max taken, m_ref moved to it, l
    // and O rescaled by exp(m_old - m_new) and P recomputed from the scores
    // still in registers. A sum of at most 2^tau keeps every P <= 2^tau (they
    // fit fp16 and bf16) and m_ref within tau of the running max. The first
    // tile always takes the max.
    // A row that has seen no key yet (every score so far masked: possible in
    // a key range of a split under the causal mask) keeps m_ref = -inf; its
    // P are computed against 0, so they are 0 (not exp2(-inf + inf)) or, if
    // the row now sees a key, large enough to take the max.
    const float2 c2 = make_float2(c, c);
    float2 se, sro;  // exact / rounded partial sums
    bool rescale_o = false;
    float alpha = 1.f;
    bool take_max = (j == 0);
    // At most two passes: the optimistic one, then (rarely) one with the max.
    for (int pass = 0; pass < 2; ++pass) {
      if (take_max) {
        // Row max with 8 independent chains of 3-input max.
        float mxa[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mxa[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
        for (int u = 16; u < C::BN; u += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mxa[i] = fmax3(mxa[i], s[u + i], s[u + 8 + i]);
        const float mx = fmaxf(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(fmax3(mxa[3], mxa[4], mxa[5]), mxa[6], mxa[7]));
        const float m_new = fmaxf(m_ref, mx * c);
        if (j > 0) {
          // = exp(m_old - m_new) in natural units; 0 for a row that saw no
          // key yet (its l and O are 0), never exp2(-inf + inf). l now, O
          // below (after P is stored, before it is released to the P.V MMA).
          alpha = m_ref > -INFINITY ? ex2_approx(m_ref - m_new) : 0.f;
          l *= alpha;
          l_o *= alpha;
          rescale_o = true;
        }
        m_ref = m_new;  // first tile: O is written fresh by the first P.V; l is 0
      }
      const float m_use = m_ref > -INFINITY ? m_ref : 0.f;
      const float2 nm2 = make_float2(-m_use, -m_use);
      se = make_float2(0.f, 0.f);
      sro = se;
#pragma unroll
      for (int q = 0; q < C::BN / 16; ++q) {
        uint32_t pk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float2 x = __ffma2_rn(make_float2(s[16 * q + 2 * u], s[16 * q + 2 * u + 1]), c2, nm2);
          const float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          se = __fadd2_rn(se, pr);
          pk[u] = pack2<BF16>(pr.x, pr.y);
          if constexpr (BF16) {
            // The two rounded values added as bf16 operands of mixed-precision
            // fp32 adds (exact conversion, one add each).
            unsigned short lo16, hi16;
            asm("mov.b32 {%0, %1}, %2;" : "=h"(lo16), "=h"(hi16) : "r"(pk[u]));
            asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(sro.x) : "h"(lo16));
            asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(sro.y) : "h"(hi16));
          }
        }
        tmem_st8(t_s + 8 * q, pk);  // keys [16q, 16q+16) -> packed columns [8q, 8q+8)
      }
      if (take_max) break;
      // The check also catches an infinite or NaN sum (a row whose P against
      // 0 overflowed after it saw no key before).
      take_max = __any_sync(0xffffffffu, !(se.x + se.y <= p_limit));
      if (!take_max) break;
      tmem_st_wait();  // this pass's P stores land before the next pass overwrites them
    }
    if (t == 0) FA_TRACE(p, kEvSm0Voted + 4 * sub, j);
    l += se.x + se.y;
    if constexpr (BF16) l_o += sro.x + sro.y;
    if (t == 0) FA_TRACE(p, kEvSm0PDone + 4 * sub, j);
    if (rescale_o) {
      // O must hold exactly tiles 0..j-1 before it is read and scaled, so
      // P(j-1) V must be complete. In this sub-tile's issue stream it is
      // followed by S(j+1), whose completion (waited for here, and then not
      // again at the top of the next tile) therefore shows it; for the last
      // tile, P(j-1) V = P(nkv-2) V is committed on its own.
      bool w;
      if (j + 1 < nkv) {
        w = wait_bar(bar128(base, C::B_SF + 2 * sub + (b ^ 1)), ((j + 1) >> 1) & 1, ctl, kWhereSFull);
        s_waited = true;
      } else {
        w = wait_bar(bar128(base, C::B_OP + sub), 0, ctl, kWhereODone);
      }
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < C::D / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(t_o + 32 * q, r);
        tmem_ld_wait();
        reg_fence(r);
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * alpha);
        tmem_st32(t_o + 32 * q, r);
      }
    }
    tmem_st_wait();
    if (t == 0) FA_TRACE(p, kEvSm0Stored + 4 * sub, j);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar128(base, C::B_PF + 2 * sub + b));
    if (t == 0) FA_TRACE(p, kEvSm0PArrive + 2 * sub, j);
#ifdef FA_TESTING
    if (p.stats_trace) {
      if (my_row < p.N) {
        float* tr = p.stats_trace + ((static_cast<size_t>(bh) * p.N + my_row) * nkv + j) * 2;
        tr[0] = m_ref * kLn2_128;
        tr[1] = l;
      }
    }
#endif
  }
  // The last P.V of this sub-tile; its commit also covers every earlier MMA of the warp.
  if (ok && nkv > 0) ok = __all_sync(0xffffffffu, wait_bar(bar128(base, C::B_OL + sub), 0, ctl, kWhereODone));
  // The whole warpgroup agrees before the epilogue, whose named barrier needs all 128 threads.
  if (!named_bar_and(1 + sub, 128, ok)) return;

  // ---- epilogue: O / l -> dtype -> swizzled staging (Q buffer) -> TMA store; LSE ----
  tc_fence_after();
  // No key to attend to (key length 0, or under the causal mask no key of
  // this split's range for this row): O = 0, LSE = -inf instead of 0/0.
  const bool empty = nkv == 0 || !(l > 0.f);
  const float inv_l = empty ? 0.f : 1.0f / (BF16 ? l_o : l);
  if (p.num_splits > 1 || p.partial) {
    // Split-KV (or one part of a merge done elsewhere): this key range's
    // normalised O (fp32) and LSE go to the partial buffers, whose rows are
    // numbered from merge_row0 (the first row of the split units; 0 unless
    // only the wave tail is split), one span per key range.
    const size_t span = static_cast<size_t>(p.B) * p.H * p.N - p.merge_row0;
    const size_t prow = static_cast<size_t>(split) * span + (static_cast<size_t>(bh) * p.N + my_row - p.merge_row0);
#pragma unroll
    for (int q = 0; q < C::D / 32; ++q) {
      uint32_t r[32];
      tmem_ld32(t_o + 32 * q, r);
      tmem_ld_wait();
      reg_fence(r);
      if (empty) {
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] = 0u;  // no key in this range: O_part = 0, LSE_part = -inf
      }
      if (my_row < p.N) {
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * C::D + 32 * q);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          dst[u] = make_float4(__uint_as_float(r[4 * u]) * inv_l, __uint_as_float(r[4 * u + 1]) * inv_l,
                               __uint_as_float(r[4 * u + 2]) * inv_l, __uint_as_float(r[4 * u + 3]) * inv_l);
      }
    }
    if (my_row < p.N) p.lse_part[prow] = empty ? -INFINITY : (m_ref + lg2_approx(l)) * kLn2_128;
    return;
  }
  const uint32_t stage = base + C::OFF_Q + sub * C::Q_SUB;
#pragma unroll
  for (int q = 0; q < C::D / 32; ++q) {
    uint32_t r[32];
    tmem_ld32(t_o + 32 * q, r);
    tmem_ld_wait();
    reg_fence(r);
    if (empty) {
#pragma unroll
      for (int u = 0; u < 32; ++u) r[u] = 0u;  // TMEM O was never written
    }
    uint32_t pk[16];
#pragma unroll
    for (int u = 0; u < 16; ++u)
      pk[u] = pack2<BF16>(__uint_as_float(r[2 * u]) * inv_l, __uint_as_float(r[2 * u + 1]) * inv_l);
    const uint32_t half = q / 2;
    const uint32_t chunk0 = (q & 1) * 4;  // 16-byte chunk within the 128-byte row
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t phys = (chunk0 + u) ^ (static_cast<uint32_t>(t) & 7u);
      const uint32_t addr = stage + half * C::Q_HALF + t * C::ROW + phys * 16;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * u]), "r"(pk[4 * u + 1]),
                   "r"(pk[4 * u + 2]), "r"(pk[4 * u + 3])
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  named_bar_sync(1 + sub, 128);
  if (t == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) tma_store_3d(&p.tm_o, stage + h * C::Q_HALF, 64 * h, row0 + C::BM * sub, bh);
    tma_store_commit();
    tma_store_wait_all();
  }
  if (my_row < p.N)
    p.lse[static_cast<size_t>(bh) * p.N + my_row] = empty ? -INFINITY : (m_ref + lg2_approx(l)) * kLn2_128;
}

template <bool BF16>
__global__ void __launch_bounds__(C128::THREADS, 1) fa_fwd_d128_kernel(const __grid_constant__ FwdParams p) {
  using C = C128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem_raw + (base - raw) + C::OFF_MISC);

  const int warp = threadIdx.x >> 5;
  // Work unit: (batch*head, 256-row Q block, key range); consecutive units
  // share a head so its K/V stay in L2 while its Q blocks are processed.
  const int nqb = (p.N + 2 * C::BM - 1) / (2 * C::BM);
  const int split = blockIdx.x % p.num_splits;
  const int qunit = p.qunit0 + blockIdx.x / p.num_splits;
  const int bh = qunit / nqb;
  // Causal, one launch over every unit unsplit: Q blocks later in the
  // sequence see more keys; they are launched first. Split launches keep the
  // natural order, in which the units of the split-KV tail plan (the last
  // ones) hold the last rows: its merge and partial buffers cover the rows
  // from merge_row0 on.
  const bool heavy_first = p.causal && p.num_splits == 1 && p.qunit_count == 0;
  const int qb = heavy_first ? nqb - 1 - qunit % nqb : qunit % nqb;
  const int row0 = qb * 2 * C::BM;
  const bool has1 = row0 + C::BM < p.N;
  // Keys this unit may see: [0, key_end); causal limits each sub-tile to its own last row.
  const int key_end = p.klen ? max(0, min(p.Nk, p.klen[bh / p.H])) : p.Nk;
  const int end0 = p.causal ? min(key_end, row0 + C::BM) : key_end;
  const int end1 = p.causal ? min(key_end, row0 + 2 * C::BM) : key_end;
  // Key ranges of a split are whole 128-key tiles of the host's plan: two of
  // this kernel's 64-key tiles each. A sub-tile whose keys end before the
  // range starts has no tile in it.
  const int range = 2 * p.split_tiles;
  const int t0 = split * range;  // first K/V tile of this key range
  const int nkv0 = max(0, min((end0 + C::BN - 1) / C::BN - t0, range));
  const int nkv1 = has1 ? max(0, min((end1 + C::BN - 1) / C::BN - t0, range)) : 0;
  const int nkv = max(nkv0, nkv1);  // tiles the producer loads

  if (threadIdx.x == 0) {
    mbar_init(bar128(base, C::B_Q), 1);
    const uint32_t nsub = has1 ? 2u : 1u;  // stage releases: one arrival per softmax warp of each sub-tile
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(bar128(base, C::B_KF + s), 1);
      mbar_init(bar128(base, C::B_KE + s), 4 * nsub);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(bar128(base, C::B_VF + s), 1);
      mbar_init(bar128(base, C::B_VE + s), 4 * nsub);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar128(base, C::B_SF + i), 1);
      mbar_init(bar128(base, C::B_PF + i), 4);  // one arrival per softmax warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar128(base, C::B_OP + i), 1);
      mbar_init(bar128(base, C::B_OL + i), 1);
      mbar_init(bar128(base, C::B_PVD + i), 1);
      mbar_init(bar128(base, C::B_DRAIN + i), 1);
    }
    misc[1] = 0;
    mbar_init_fence();
  }
  if (warp == C::WARP_MMA0) {
    tmem_alloc(base + C::OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const WaitCtl ctl{p, base + C::OFF_MISC + 4};  // misc[1] is the abort flag
  if (threadIdx.x == 0) FA_TRACE(p, kEvCta, 0);

  if (warp >= 8) {
    if (warp == C::WARP_TMA) {
      if ((threadIdx.x & 31) == 0) producer128(p, base, bh, row0, nkv0, nkv1, t0, ctl);
      __syncwarp();
    } else if (warp == C::WARP_MMA0) {
      mma128<BF16, 0>(p, base, tmem, nkv0, ctl);
      __syncwarp();
    } else if (warp == C::WARP_MMA1 && has1) {
      mma128<BF16, 1>(p, base, tmem, nkv1, ctl);
      __syncwarp();
    }
  } else {
    const int sub = warp / 4;
    if (sub == 0 || has1) softmax128<BF16>(p, base, tmem, sub, bh, row0, split, t0, sub ? nkv1 : nkv0, key_end, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    FA_TRACE(p, kEvCta, 1);
#ifdef FA_TESTING
    if (p.timeline && blockIdx.x < kTraceCtas) {
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      p.timeline[(static_cast<size_t>(blockIdx.x) * kTraceEvents + kEvCta) * kTraceTiles + 2] = smid;
    }
#endif
  }
  if (warp == C::WARP_MMA0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <bool BF16>
cudaError_t launch128(const FwdParams& p, cudaStream_t stream) {
  using C = C128;
  auto kern = fa_fwd_d128_kernel<BF16>;
  static std::atomic<uint64_t> attr_done{0};  // one bit per device ordinal (< 64)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit);
  }
  const long long all_qunits = static_cast<long long>(p.B) * p.H * ((p.N + 2 * C::BM - 1) / (2 * C::BM));
  const long long qunits = p.qunit_count > 0 ? p.qunit_count : all_qunits;
  if (p.qunit0 < 0 || p.qunit0 + qunits > all_qunits) return cudaErrorInvalidValue;
  const long long units = qunits * p.num_splits;
  if (units <= 0 || units > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<dim3(static_cast<unsigned>(units)), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d128(const FwdParams& p, bool bf16, cudaStream_t stream) {
  return bf16 ? launch128<true>(p, stream) : launch128<false>(p, stream);
}

}  // namespace fa
