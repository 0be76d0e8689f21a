// fa_bwd_f16.cu — FlashAttention backward pass (dQ, dK, dV) for fp16 / bf16 on sm_103a.
//
// Algorithm: backward by recomputation (the MUSA SDK guide's fourth core
// principle, "重计算（Recompute）换存储"; the Triton page, sections 2.4 and 4.4:
// P is not stored by the forward pass; it is rebuilt from Q, K and the saved
// row statistics, and the chain rule is applied tile by tile). With
// LSE_i = ln sum_j exp(s_ij) from the forward pass and D_i = sum_c dO_ic O_ic:
//     P_ij  = exp(s_ij - LSE_i),        s_ij = scale * q_i . k_j
//     dV_j  = sum_i P_ij dO_i
//     dS_ij = P_ij (dO_i . v_j - D_i)
//     dQ_i  = scale * sum_j dS_ij k_j,  dK_j = scale * sum_i dS_ij q_i
// Like the forward pass, no N x N matrix reaches HBM.
//
// Three kernels:
//   fa_bwd_pre   per row: D_i (fp32), LSE_i * log2(e), and a zeroed fp32 dQ
//                accumulator row; rows past N of the last tile get D = 0 and
//                LSE * log2(e) = +inf, so their P is exactly 0
//   fa_bwd_main  one CTA per (batch*head, 128-key tile): K_j and V_j stay in
//                shared memory, dK_j and dV_j accumulate in TMEM over all Q
//                tiles; each Q tile's dQ contribution is added into the fp32
//                accumulator with TMA reduce-add
//   fa_bwd_post  dQ = accumulator rounded to the input type
//
// fa_bwd_main on GB300 (16 warps; TMEM lanes are keys for S^T, dP^T, dV, dK
// and queries for dQ):
//   warp 12     TMA producer: K_j, V_j once; Q_i (+ its LSE and D rows) into a
//               2-stage ring; dO_i into a 1-stage (d=128) / 2-stage (d=64) ring
//   warps 13-14 MMA warps (one elected lane issues), per Q tile i:
//                 S^T  = K_j Q_i^T   (SS)           -> TMEM [0,128)
//                 dP^T = V_j dO_i^T  (SS)           -> TMEM [128,256)
//                 dV  += P^T dO_i    (TS: P^T from TMEM, dO MN-major)
//                 dK  += dS^T Q_i    (SS: dS^T from SMEM, Q MN-major)
//                 dQ_i = dS K_j      (SS: dS^T read MN-major, K MN-major)
//               warp 13 issues dQ_i, dK_i as soon as dS_i is formed; warp 14
//               issues dP^T_{i+1}, dV_{i+1}, S^T_{i+2}, so that S^T_{i+2} runs
//               while dS_{i+1} is formed and each warp's waits and commits
//               overlap the other's MMAs
//   warps 0-3   queries 0-63 of every Q tile, warps 4-7 queries 64-127 (one
//   and 4-7     thread per key): P = 2^(s*scale*log2e - LSE*log2e) in fp32,
//               written back as 16-bit pairs over S^T columns [0,32) / [64,96)
//               for the dV product and kept as fp32 P*scale in registers;
//               dS^T*scale = P*scale (dP^T - D) rounded to 16 bits into their
//               half of the dS^T tile in SMEM; at the end dV_j / dK_j
//   warps 8-11  dQ (one thread per query): all d columns of dQ_i from TMEM
//               into registers (which frees the columns at once), then
//               32-column fp32 boxes through two SMEM buffers into TMA
//               reduce-adds on the accumulator. The reduce-adds (64 KB per Q
//               tile for d=128) drain at the SM's write rate to L2, so they
//               run beside the other roles instead of in their chain.
//   warp 15     idle (completes the fourth warpgroup)
// Registers: launched at 128 per thread; warpgroups 0-2 grow to 160 / 160 /
// 144 and warpgroup 3 shrinks to 48 (setmaxnreg).
// TMEM (512 columns): S^T [0,128), dP^T [128,256), dV [256,256+d),
// dK [256+d,256+2d); dQ_i reuses the dP^T columns for d=128 (dP^T_i is
// consumed once dS_i is written; dP^T_{i+1} waits for the read-out of dQ_i)
// and has [384,448) for d=64.
// S^T_{i+1} overwrites P^T_i: it is issued behind dV_i by the same warp and
// one CTA's MMAs execute in issue order (-DFA_STRICT_MMA_ORDER waits for dV_i
// to complete instead).
#include <atomic>
#include <type_traits>

#include <cuda_fp16.h>

#include "fa_bwd_order.cuh"
#include "fa_device_common.cuh"

namespace fa {
namespace {

constexpr float kLog2eB = 1.4426950408889634f;

template <int D>
struct BCfg {
  static constexpr int BQ = 128;                    // queries per Q tile (MMA N of S^T)
  static constexpr int BK = 128;                    // keys per CTA (TMEM lanes, MMA M)
  static constexpr int QST = (D == 128) ? 2 : 3;    // Q (+ LSE, D rows) stages
  static constexpr int OST = (D == 128) ? 1 : 2;    // dO stages
  static constexpr uint32_t ROW = 128;              // bytes of one 128-byte swizzle row (64 16-bit elements)
  static constexpr uint32_t TILE = 128 * D * 2;     // a 128-row tile of Q, K, V or dO
  static constexpr uint32_t HALF = 128 * ROW;       // one 64-column half of a tile
  static constexpr uint32_t DS_BYTES = 128 * 128 * 2;
  static constexpr uint32_t BOX = 128 * 128;        // one fp32 dQ box: 128 rows x 32 columns
  static constexpr int NBOX = D / 32;               // dQ boxes per Q tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TILE;
  static constexpr uint32_t OFF_Q = OFF_V + TILE;
  static constexpr uint32_t OFF_DO = OFF_Q + QST * TILE;
  static constexpr uint32_t OFF_DS = OFF_DO + OST * TILE;
  static constexpr uint32_t OFF_DQS = OFF_DS + DS_BYTES;   // two dQ staging boxes
  static constexpr uint32_t OFF_ROWS = OFF_DQS + 2 * BOX;  // [QST] x {lse2[128], dsum[128]} fp32
  static constexpr uint32_t ROWS_BYTES = 2 * 128 * 4;
  static constexpr uint32_t OFF_BAR = OFF_ROWS + QST * ROWS_BYTES;
  static constexpr int B_K = 0, B_V = 1;
  static constexpr int B_QF = 2, B_QE = B_QF + QST;
  static constexpr int B_OF = B_QE + QST, B_OE = B_OF + OST;
  static constexpr int B_SF = B_OE + OST, B_DPF = B_SF + 1, B_PF = B_DPF + 1, B_DSF = B_PF + 1;
  static constexpr int B_DQF = B_DSF + 1, B_DQE = B_DQF + 1, B_DSE = B_DQE + 1, B_DONE = B_DSE + 1;
  static constexpr int NBAR = B_DONE + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  // The dynamic shared memory starts 1 KB-aligned (checked in the kernel): no slack.
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  static constexpr uint32_t T_DQ = (D == 128) ? 128 : 384;
  static constexpr int THREADS = 512;
  static constexpr int WARP_TMA = 12, WARP_MMA = 13, WARP_MMA_SP = 14;
  static constexpr int LAUNCH_REGS = 128, SM_REGS = 160, DQ_REGS = 144, LOW_REGS = 48;
  static_assert(128 * (2 * SM_REGS + DQ_REGS + LOW_REGS) <= THREADS * LAUNCH_REGS, "register split exceeds the pool");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(OFF_DS % 1024 == 0 && OFF_DO % 1024 == 0 && OFF_Q % 1024 == 0, "swizzled buffers need 1 KB alignment");
};

using BCtl = WaitCtlT<BwdParams>;

template <int D>
__device__ __forceinline__ uint32_t bbar(uint32_t base, int i) {
  return base + BCfg<D>::OFF_BAR + 8u * i;
}

// --------------------------------------------------------------------------
// TMA producer (one thread)
// --------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void bwd_producer(const BwdParams& p, uint32_t base, int bh, int kv0, int q_first,
                                             int nq, const BCtl& ctl) {
  using C = BCfg<D>;
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);
  tma_prefetch_desc(&p.tm_do);
  const uint32_t bk = bbar<D>(base, C::B_K), bv = bbar<D>(base, C::B_V);
  mbar_arrive_expect_tx(bk, C::TILE);
#pragma unroll
  for (int h = 0; h < D / 64; ++h) tma_load_3d(base + C::OFF_K + h * C::HALF, &p.tm_k, bk, 64 * h, kv0, bh);
  mbar_arrive_expect_tx(bv, C::TILE);
#pragma unroll
  for (int h = 0; h < D / 64; ++h) tma_load_3d(base + C::OFF_V + h * C::HALF, &p.tm_v, bv, 64 * h, kv0, bh);

  const size_t row_base = static_cast<size_t>(bh) * p.n_pad;
  int nqi = 0, noi = 0;  // Q / dO tiles whose loads were issued
  bool ok = true;
  for (int i = 0; i < nq; ++i) {
    const int qs = i % C::QST;
    if (!wait_bar(bbar<D>(base, C::B_QE + qs), ((i / C::QST) & 1) ^ 1, ctl, kWhereBwdQEmpty)) { ok = false; break; }
    const uint32_t qf = bbar<D>(base, C::B_QF + qs);
    mbar_arrive_expect_tx(qf, C::TILE + C::ROWS_BYTES);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_load_3d(base + C::OFF_Q + qs * C::TILE + h * C::HALF, &p.tm_q, qf, 64 * h, (q_first + i) * C::BQ, bh);
    const uint32_t rows = base + C::OFF_ROWS + qs * C::ROWS_BYTES;
    bulk_load(rows, p.lse2 + row_base + static_cast<size_t>(q_first + i) * C::BQ, 512, qf);
    bulk_load(rows + 512, p.dsum + row_base + static_cast<size_t>(q_first + i) * C::BQ, 512, qf);
    nqi = i + 1;
    FA_TRACE(p, kBvQLoad, i);
#ifdef FA_TESTING
    if (p.inject == 1 && i == 0) continue;  // fault injection: dO_0 is never loaded
#endif
    const int os = i % C::OST;
    if (!wait_bar(bbar<D>(base, C::B_OE + os), ((i / C::OST) & 1) ^ 1, ctl, kWhereBwdDoEmpty)) { ok = false; break; }
    const uint32_t of = bbar<D>(base, C::B_OF + os);
    mbar_arrive_expect_tx(of, C::TILE);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_load_3d(base + C::OFF_DO + os * C::TILE + h * C::HALF, &p.tm_do, of, 64 * h, (q_first + i) * C::BQ, bh);
    noi = i + 1;
    FA_TRACE(p, kBvDOLoad, i);
  }
  // Drain, always (the loop ended, this thread's wait gave up, or another role
  // may abort later): every copy this thread started must land before the CTA
  // exits. Cheap when nothing failed: the consumers need these copies anyway.
  (void)ok;
  {
    wait_bar_drain(bk, 0, ctl);
    wait_bar_drain(bv, 0, ctl);
    for (int t = nqi > C::QST ? nqi - C::QST : 0; t < nqi; ++t)
      wait_bar_drain(bbar<D>(base, C::B_QF + t % C::QST), (t / C::QST) & 1, ctl);
    for (int t = noi > C::OST ? noi - C::OST : 0; t < noi; ++t) {
#ifdef FA_TESTING
      if (p.inject == 1 && t == 0) continue;  // never armed
#endif
      wait_bar_drain(bbar<D>(base, C::B_OF + t % C::OST), (t / C::OST) & 1, ctl);
    }
  }
}

// --------------------------------------------------------------------------
// MMA warp (whole warp; one elected lane issues)
// --------------------------------------------------------------------------
// A descriptor the compiler must treat as computed here: the k-loops below are
// unrolled (back-to-back MMAs issue at the full rate only from straight-line
// code), and without this the compiler hoists every k-step's descriptor of all
// five products out of the Q-tile loop into registers the warp does not have.
__device__ __forceinline__ uint64_t opaque(uint64_t x) {
  asm volatile("" : "+l"(x));
  return x;
}

// 128 x 128 x D product of two K-major tiles (both 64-column halves, 128-byte swizzle).
template <int D>
__device__ __forceinline__ void mma_kmajor_tiles(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
  const uint64_t a0 = opaque(smem_desc_sw128(a_base, 16, 1024));
  const uint64_t b0 = opaque(smem_desc_sw128(b_base, 16, 1024));
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk / 4) * BCfg<D>::HALF + (kk & 3) * 32u) >> 4;
    mma_f16_ss_elect(d_tmem, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// Two MMA warps feed the one tensor pipe, so that the waits and commits of
// one (each leaves the pipe idle for about a hundred cycles when nothing else
// is queued: it holds about one MMA) overlap the other's MMAs:
//   warp 13: dQ_i, dK_i                  (both need dS_i)
//   warp 14: S^T_0, dP^T_0, dV_0, S^T_1, then dP^T_{i+1}, dV_{i+1}, S^T_{i+2}
// Each keeps its own products in order (S^T_{i+2} overwrites P^T_{i+1} right
// behind dV_{i+1} in warp 14); everything between the two warps goes through
// mbarriers.
template <int D, bool BF16>
struct BwdMma {
  using C = BCfg<D>;
  static constexpr uint32_t fmt = BF16 ? 1u : 0u;
  static constexpr uint32_t idesc_st = make_idesc(fmt, 0, 0, 128, 128);  // S^T, dP^T: M = keys, N = queries
  static constexpr uint32_t idesc_acc = make_idesc(fmt, 0, 1, 128, D);   // dV, dK: B (dO, Q) has d contiguous
  static constexpr uint32_t idesc_dq = make_idesc(fmt, 1, 1, 128, D);    // dQ: A = dS read M-major, B = K
  // MN-major operands: 16 K-rows = two 8-row swizzle atoms (2048 bytes); the
  // 64-wide MN blocks are LBO apart (a tile's halves; the dS^T halves for A).
  static constexpr uint32_t lbo_d = (D == 64) ? 1024u : C::HALF;
};

// Warp 13: the two products that need dS_i.
template <int D, bool BF16>
__device__ __forceinline__ void bwd_mma_dsdep(const BwdParams& p, uint32_t base, uint32_t tmem, int nq,
                                              const BCtl& ctl) {
  using C = BCfg<D>;
  using M = BwdMma<D, BF16>;
  const uint32_t b_dsf = bbar<D>(base, C::B_DSF), b_dqf = bbar<D>(base, C::B_DQF), b_dqe = bbar<D>(base, C::B_DQE);
  const uint32_t b_dse = bbar<D>(base, C::B_DSE), b_done = bbar<D>(base, C::B_DONE);
  const uint64_t dq_a0 = smem_desc_sw128(base + C::OFF_DS, C::HALF, 1024);
  const uint64_t dq_b0 = smem_desc_sw128(base + C::OFF_K, M::lbo_d, 1024);
  const uint64_t dk_a0 = smem_desc_sw128(base + C::OFF_DS, 16, 1024);
  for (int i = 0; i < nq; ++i) {
    if (!wait_bar_warp(b_dsf, i & 1, ctl, kWhereBwdDsFull)) break;
    if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvDQReady, i);
    if constexpr (D == 64) {
      // dQ_{i-1} must have left its TMEM columns.
      if (i > 0 && !wait_bar_warp(b_dqe, (i - 1) & 1, ctl, kWhereBwdDqEmpty)) break;
    }
    tc_fence_after();
    {
      const uint64_t a0 = opaque(dq_a0), b0 = opaque(dq_b0);
#pragma unroll
      for (int kk = 0; kk < C::BK / 16; ++kk)
        mma_f16_ss_elect(tmem + C::T_DQ, a0 + ((kk * 2048u) >> 4), b0 + ((kk * 2048u) >> 4), M::idesc_dq,
                         kk > 0 ? 1u : 0u);
    }
    tc_commit_elect(b_dqf);
    if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvDQ, i);
    {
      const uint64_t b0 = opaque(smem_desc_sw128(base + C::OFF_Q + (i % C::QST) * C::TILE, M::lbo_d, 1024));
      const uint64_t a0 = opaque(dk_a0);
#pragma unroll
      for (int kk = 0; kk < C::BQ / 16; ++kk) {
        const uint32_t aoff = ((kk / 4) * C::HALF + (kk & 3) * 32u) >> 4;
        mma_f16_ss_elect(tmem + C::T_DK, a0 + aoff, b0 + ((kk * 2048u) >> 4), M::idesc_acc,
                         (i > 0 || kk > 0) ? 1u : 0u);
      }
    }
    tc_commit_elect(bbar<D>(base, C::B_QE + i % C::QST));  // Q_i (and its rows) are free once dK_i is done
    tc_commit_elect(b_dse);                                // so is the dS^T tile (dQ_i was issued before)
    if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvDK, i);
  }
  // One commit after this warp's last MMA (the barrier counts both MMA warps):
  // the epilogues wait for it, and every MMA completes before TMEM is freed.
  tc_commit_elect(b_done);
  __all_sync(0xffffffffu, wait_bar_drain(b_done, 0, ctl));
}

// Warp 14: S^T, dP^T and dV.
template <int D, bool BF16>
__device__ __forceinline__ void bwd_mma_sp(const BwdParams& p, uint32_t base, uint32_t tmem, int nq,
                                           const BCtl& ctl) {
  using C = BCfg<D>;
  using M = BwdMma<D, BF16>;
  const uint32_t b_sf = bbar<D>(base, C::B_SF), b_dpf = bbar<D>(base, C::B_DPF);
  const uint32_t b_pf = bbar<D>(base, C::B_PF), b_dsf = bbar<D>(base, C::B_DSF);
  const uint32_t b_dqe = bbar<D>(base, C::B_DQE), b_done = bbar<D>(base, C::B_DONE);

  // S^T_j = K Q_j^T into the S^T columns, over P^T_{j-1}, whose dV_{j-1} is issued before.
  auto issue_s = [&](int j) {
    mma_kmajor_tiles<D>(tmem + C::T_S, base + C::OFF_K, base + C::OFF_Q + (j % C::QST) * C::TILE, M::idesc_st);
    tc_commit_elect(b_sf);
  };
  // dP^T_j = V dO_j^T
  auto issue_dp = [&](int j) {
    mma_kmajor_tiles<D>(tmem + C::T_DP, base + C::OFF_V, base + C::OFF_DO + (j % C::OST) * C::TILE, M::idesc_st);
    tc_commit_elect(b_dpf);
  };
  // dV += P^T_j dO_j (K = the 128 queries of tile j). P^T of queries 0-63 is
  // packed in S^T columns [0,32), of queries 64-127 in [64,96). dO_j is free
  // afterwards (its dP^T_j was issued before).
  auto issue_dv = [&](int j) {
    const uint64_t b0 = opaque(smem_desc_sw128(base + C::OFF_DO + (j % C::OST) * C::TILE, M::lbo_d, 1024));
#pragma unroll
    for (int kk = 0; kk < C::BQ / 16; ++kk)
      mma_f16_ts_elect(tmem + C::T_DV, tmem + C::T_S + (kk < 4 ? 8 * kk : 64 + 8 * (kk - 4)),
                       b0 + ((kk * 2048u) >> 4), M::idesc_acc, (j > 0 || kk > 0) ? 1u : 0u);
    tc_commit_elect(bbar<D>(base, C::B_OE + j % C::OST));
  };

  if (!wait_bar_warp(bbar<D>(base, C::B_K), 0, ctl, kWhereBwdKV)) goto drain;
  if (!wait_bar_warp(bbar<D>(base, C::B_QF), 0, ctl, kWhereBwdQFull)) goto drain;
  tc_fence_after();
  issue_s(0);
  if (!wait_bar_warp(bbar<D>(base, C::B_V), 0, ctl, kWhereBwdKV)) goto drain;
  if (!wait_bar_warp(bbar<D>(base, C::B_OF), 0, ctl, kWhereBwdDoFull)) goto drain;
  tc_fence_after();
  issue_dp(0);
  if (!wait_bar_warp(b_pf, 0, ctl, kWhereBwdPFull)) goto drain;
  tc_fence_after();
  issue_dv(0);
  if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvDV, 0);
  if (nq > 1) {
#ifdef FA_STRICT_MMA_ORDER
    if (!wait_bar_warp(bbar<D>(base, C::B_OE), 0, ctl, kWhereBwdDoEmpty)) goto drain;
#endif
    if (!wait_bar_warp(bbar<D>(base, C::B_QF + 1 % C::QST), (1 / C::QST) & 1, ctl, kWhereBwdQFull)) goto drain;
    tc_fence_after();
    issue_s(1);
  }
  for (int i = 0; i + 1 < nq; ++i) {
    const int n1 = i + 1;
    // dP^T_{i+1} overwrites the dP^T columns: the softmax warps must be done with
    // dP^T_i, and for d = 128 the dQ warps with dQ_i (which implies the former).
    if constexpr (D == 128) {
      if (!wait_bar_warp(b_dqe, i & 1, ctl, kWhereBwdDqEmpty)) goto drain;
    } else {
      if (!wait_bar_warp(b_dsf, i & 1, ctl, kWhereBwdDsFull)) goto drain;
    }
    if (!wait_bar_warp(bbar<D>(base, C::B_OF + n1 % C::OST), (n1 / C::OST) & 1, ctl, kWhereBwdDoFull)) goto drain;
    if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvDPReady, n1);
    tc_fence_after();
    issue_dp(n1);
    if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvDP, n1);
    if (!wait_bar_warp(b_pf, n1 & 1, ctl, kWhereBwdPFull)) goto drain;
    if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvDVReady, n1);
    tc_fence_after();
    issue_dv(n1);
    if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvDV, n1);
    if (i + 2 < nq) {
      const int n2 = i + 2;
#ifdef FA_STRICT_MMA_ORDER
      // dV_{i+1} complete before S^T_{i+2} reuses the P^T columns.
      if (!wait_bar_warp(bbar<D>(base, C::B_OE + n1 % C::OST), (n1 / C::OST) & 1, ctl, kWhereBwdDoEmpty))
        goto drain;
#endif
      if (!wait_bar_warp(bbar<D>(base, C::B_QF + n2 % C::QST), (n2 / C::QST) & 1, ctl, kWhereBwdQFull)) goto drain;
      if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvSReady, n2);
      tc_fence_after();
      issue_s(n2);
      if (threadIdx.x % 32 == 0) FA_TRACE(p, kBvS, n2);
    }
  }
drain:
  tc_commit_elect(b_done);
  __all_sync(0xffffffffu, wait_bar_drain(b_done, 0, ctl));
}

// Store a 128 x D fp32 TMEM accumulator (this thread's lane = row t) as a
// 16-bit tile through the swizzled staging buffer `stage` with TMA.
template <int D, bool BF16>
__device__ __forceinline__ void store_acc_tile(uint32_t t_acc, uint32_t stage, int t, int bar_id,
                                               const CUtensorMap* map, int row0, int bh) {
  using C = BCfg<D>;
#pragma unroll
  for (int q = 0; q < D / 32; ++q) {
    uint32_t r[32];
    tmem_ld32(t_acc + 32 * q, r);
    tmem_ld_wait();
    reg_fence(r);
    uint32_t pk[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) pk[u] = pack2<BF16>(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
    const uint32_t half = q / 2, chunk0 = (q & 1) * 4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t phys = (chunk0 + u) ^ (static_cast<uint32_t>(t) & 7u);
      const uint32_t addr = stage + half * C::HALF + t * C::ROW + phys * 16;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * u]), "r"(pk[4 * u + 1]),
                   "r"(pk[4 * u + 2]), "r"(pk[4 * u + 3])
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  named_bar_sync(bar_id, 128);
  if (t == 0) {
#pragma unroll
    for (int h = 0; h < D / 64; ++h) tma_store_3d(map, stage + h * C::HALF, 64 * h, row0, bh);
    tma_store_commit();
    tma_store_wait_all();
  }
}

// --------------------------------------------------------------------------
// Softmax warpgroup W (warps 4W .. 4W+3): queries [64W, 64W+64) of P^T and
// dS^T; at the end dV (W = 0) or dK (W = 1)
// --------------------------------------------------------------------------
// FULL: no entry of any tile is masked (no causal mask, no key lengths, N a
// multiple of 128): only the unmasked copy of the P loop is compiled.
template <int D, bool BF16, int W, bool FULL>
__device__ __forceinline__ void bwd_softmax(const BwdParams& p, uint8_t* smem, uint32_t base, uint32_t tmem, int bh,
                                            int kv0, int nq, int key_end, const BCtl& ctl) {
  using C = BCfg<D>;
  constexpr int BAR = 1 + W;  // this warpgroup's named barrier
  const int t = threadIdx.x - 128 * W;  // key row = TMEM lane
  const int lane = t & 31;
  const uint32_t lane_base = static_cast<uint32_t>(t & ~31) << 16;
  const uint32_t t_s = tmem + lane_base + C::T_S + 64 * W, t_dp = tmem + lane_base + C::T_DP + 64 * W;
  const float c = p.scale * kLog2eB;
  // Masks. Keys at or past key_end (past N, or past the batch's key length)
  // get P = 0 in every Q tile; with the causal mask the first Q tile is the
  // diagonal one (same rows as the keys) and query c of it sees key t only if
  // c >= t. For this thread: P of query column c (0..63 of this half) is 0
  // when c < lim. A tile with no masked entry skips the test.
  const bool key_ok = kv0 + t < key_end;
  const int lim_diag = key_ok ? t - 64 * W : 64;
  const int lim_rest = key_ok ? 0 : 64;
  const bool rest_masked = kv0 + C::BK > key_end;
  const float2 c2 = make_float2(c, c);
  const float2 sc2 = make_float2(p.scale, p.scale);
  const uint32_t b_sf = bbar<D>(base, C::B_SF), b_dpf = bbar<D>(base, C::B_DPF);
  const uint32_t b_pf = bbar<D>(base, C::B_PF), b_dsf = bbar<D>(base, C::B_DSF);
  const uint32_t b_dse = bbar<D>(base, C::B_DSE);
  // Row t of this warpgroup's half of dS^T (128-byte swizzle: 16-byte chunk c sits at c ^ (t & 7)).
  uint4* ds_row = reinterpret_cast<uint4*>(smem + C::OFF_DS + W * C::HALF + t * C::ROW);
  bool ok = true;
  float ps[64];  // P*scale of this thread's key for queries [64W, 64W+64) of the current tile

  // Each wait is agreed by the warp (its TMEM accesses are per warp), not by
  // the warpgroup: a warp that gives up leaves the loop, the others give up
  // too once the abort flag is raised (the MMA warps then wait in vain for its
  // arrivals), and all four meet once, at the agreement before the epilogue,
  // whose named barriers need all 128 threads.
  for (int i = 0; i < nq; ++i) {
    // lse2[128], dsum[128] of Q tile i, read as plain shared-memory loads (the compiler schedules them freely)
    const float4* lse4 = reinterpret_cast<const float4*>(smem + C::OFF_ROWS + (i % C::QST) * C::ROWS_BYTES) + 16 * W;
    const float4* dsum4 = lse4 + 32;
    // ---- P_i: S^T columns -> fp32 P (kept, times scale) and 16-bit P^T in TMEM
    if (!__all_sync(0xffffffffu, wait_bar(b_sf, i & 1, ctl, kWhereBwdSFull))) { ok = false; break; }
    if (W == 0 && t == 0) FA_TRACE(p, kBvSmS, i);
    tc_fence_after();
    uint32_t rs[2][32];
    tmem_ld32(t_s, rs[0]);
    tmem_ld32(t_s + 32, rs[1]);
    tmem_ld_wait();
    reg_fence(rs[0]);
    reg_fence(rs[1]);
    // Two copies of the P loop: the masked one only for tiles with a masked entry.
    auto p_phase = [&](auto mask_tag, int lim) {
      constexpr bool kMasked = decltype(mask_tag)::value;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t (&r)[32] = rs[q];
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 l4 = lse4[8 * q + u];
          const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1])), c2,
                                       make_float2(-l4.x, -l4.y));
          const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])),
                                       c2, make_float2(-l4.z, -l4.w));
          float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
          float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
          if constexpr (kMasked) {
            const int c0 = 32 * q + 4 * u;
            if (c0 < lim) p0.x = 0.f;
            if (c0 + 1 < lim) p0.y = 0.f;
            if (c0 + 2 < lim) p1.x = 0.f;
            if (c0 + 3 < lim) p1.y = 0.f;
          }
          pk[2 * u] = pack2<BF16>(p0.x, p0.y);
          pk[2 * u + 1] = pack2<BF16>(p1.x, p1.y);
          const float2 s0 = __fmul2_rn(p0, sc2), s1 = __fmul2_rn(p1, sc2);
          ps[32 * q + 4 * u] = s0.x;
          ps[32 * q + 4 * u + 1] = s0.y;
          ps[32 * q + 4 * u + 2] = s1.x;
          ps[32 * q + 4 * u + 3] = s1.y;
        }
        // Queries [32q, 32q+32) of this half -> packed columns [16q, 16q+16) (both chunks were read above).
        tmem_st16(t_s + 16 * q, pk);
        if (q == 0 && W == 0 && t == 0) FA_TRACE(p, kBvSmPChunk0, i);
      }
    };
    if constexpr (FULL) {
      p_phase(std::false_type{}, 0);
    } else {
      const bool diag = p.causal && i == 0;
      if (diag || rest_masked)
        p_phase(std::true_type{}, diag ? lim_diag : lim_rest);
      else
        p_phase(std::false_type{}, 0);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(b_pf);
    if (t == 0) FA_TRACE(p, W == 0 ? kBvSmP : kBvW1P, i);

    // ---- dS_i: dS^T * scale = P*scale (dP^T - D), 16-bit, into row t of this warpgroup's dS^T half
    if (!__all_sync(0xffffffffu, wait_bar(b_dpf, i & 1, ctl, kWhereBwdDpFull))) { ok = false; break; }
    if (W == 0 && t == 0) FA_TRACE(p, kBvSmDp, i);
    // dS^T_{i-1} is read by dQ_{i-1} and dK_{i-1}, issued before dP^T_i: this
    // wait is normally over by now.
    if (i > 0 && !__all_sync(0xffffffffu, wait_bar(b_dse, (i - 1) & 1, ctl, kWhereBwdDsEmpty))) { ok = false; break; }
    if (W == 0 && t == 0) FA_TRACE(p, kBvSmDsWaited, i);
    tc_fence_after();
    uint32_t rdp[2][32];
    tmem_ld32(t_dp, rdp[0]);
    tmem_ld32(t_dp + 32, rdp[1]);
    tmem_ld_wait();
    reg_fence(rdp[0]);
    reg_fence(rdp[1]);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t (&r)[32] = rdp[q];
      uint32_t pk[16];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 d4 = dsum4[8 * q + u];
        const float2 e0 = __fadd2_rn(make_float2(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1])),
                                     make_float2(-d4.x, -d4.y));
        const float2 e1 = __fadd2_rn(make_float2(__uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])),
                                     make_float2(-d4.z, -d4.w));
        const float2 g0 = __fmul2_rn(e0, make_float2(ps[32 * q + 4 * u], ps[32 * q + 4 * u + 1]));
        const float2 g1 = __fmul2_rn(e1, make_float2(ps[32 * q + 4 * u + 2], ps[32 * q + 4 * u + 3]));
        pk[2 * u] = pack2<BF16>(g0.x, g0.y);
        pk[2 * u + 1] = pack2<BF16>(g1.x, g1.y);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t phys = (4 * q + u) ^ (static_cast<uint32_t>(t) & 7u);
        ds_row[phys] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      if (W == 0 && t == 0) FA_TRACE(p, q == 0 ? kBvSmDsChunk0 : kBvSmDsChunk1, i);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(b_dsf);
    if (t == 0) FA_TRACE(p, W == 0 ? kBvSmDs : kBvW1Ds, i);
  }
  if (ok) ok = wait_bar(bbar<D>(base, C::B_DONE), 0, ctl, kWhereBwdDone);
  if (!named_bar_and(BAR, 128, ok)) return;
  tc_fence_after();
  // dV_j (W = 0) or dK_j (W = 1; the scale is already in dS) -> 16-bit, staged in Q stage W.
  if constexpr (W == 0)
    store_acc_tile<D, BF16>(tmem + lane_base + C::T_DV, base + C::OFF_Q, t, BAR, &p.tm_dv, kv0, bh);
  else
    store_acc_tile<D, BF16>(tmem + lane_base + C::T_DK, base + C::OFF_Q + C::TILE, t, BAR, &p.tm_dk, kv0, bh);
}

// --------------------------------------------------------------------------
// dQ warpgroup (warps 8-11): dQ_i -> registers -> fp32 boxes -> TMA reduce-add
// --------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void bwd_dq(const BwdParams& p, uint32_t base, uint32_t tmem, int bh, int q_first,
                                       int nq, const BCtl& ctl) {
  using C = BCfg<D>;
  constexpr int BAR = 3;
  const int t = threadIdx.x - 256;  // query row within the Q tile = TMEM lane
  const int lane = t & 31;
  const uint32_t t_dq = tmem + (static_cast<uint32_t>(t & ~31) << 16) + C::T_DQ;
  const uint32_t b_dqf = bbar<D>(base, C::B_DQF), b_dqe = bbar<D>(base, C::B_DQE);
  for (int i = 0; i < nq; ++i) {
    // Agreed by the whole warpgroup: the named barriers below need all 128 threads.
    if (!named_bar_and(BAR, 128, wait_bar(b_dqf, i & 1, ctl, kWhereBwdDqFull))) break;
    if (t == 0) FA_TRACE(p, kBvSmDq, i);
    tc_fence_after();
    uint32_t r[C::NBOX][32];
#pragma unroll
    for (int b = 0; b < C::NBOX; ++b) tmem_ld32(t_dq + 32 * b, r[b]);
    tmem_ld_wait();
#pragma unroll
    for (int b = 0; b < C::NBOX; ++b) reg_fence(r[b]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(b_dqe);  // the MMA warp may reuse these TMEM columns
    if (t == 0) FA_TRACE(p, kBvSmDqLoaded, i);
#pragma unroll
    for (int b = 0; b < C::NBOX; ++b) {
      const uint32_t buf = base + C::OFF_DQS + (b & 1) * C::BOX;
      // The reduce-add that last read this buffer is the one before the most recent.
      if (t == 0) bulk_wait_read<1>();
      named_bar_sync(BAR, 128);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t phys = static_cast<uint32_t>(u) ^ (static_cast<uint32_t>(t) & 7u);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + t * 128u + phys * 16), "r"(r[b][4 * u]),
                     "r"(r[b][4 * u + 1]), "r"(r[b][4 * u + 2]), "r"(r[b][4 * u + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      named_bar_sync(BAR, 128);
      if (t == 0) {
        tma_reduce_add_3d(&p.tm_dqacc, buf, 32 * b, (q_first + i) * C::BQ, bh);
        tma_store_commit();
      }
    }
    if (t == 0) FA_TRACE(p, kBvSmRed, i);
  }
  if (t == 0) tma_store_wait_all();  // every reduce-add is complete before the CTA exits
}

template <int D, bool BF16, bool FULL>
__global__ void __launch_bounds__(BCfg<D>::THREADS, 1) fa_bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using C = BCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    // The layout assumes a 1 KB-aligned start (there is no room for slack):
    // report it and leave before anything is set up.
    if (threadIdx.x == 0) atomicOr(p.status, kStatusSmemAlign);
    return;
  }
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem_raw + C::OFF_MISC);
  const int warp = threadIdx.x >> 5;
  // This CTA's head and key tile (fa_bwd_order.cuh: a head's key tiles in a
  // row; with the causal mask, longest first within windows of heads).
  const int nt = (p.N + C::BK - 1) / C::BK;
  const BwdTileOf tile = bwd_tile_of(static_cast<int>(blockIdx.x), p.B * p.H, nt, p.N, D, p.causal != 0);
  const int bh = tile.bh;
  const int kv0 = tile.kt * C::BK;
  int key_end = p.N;
  if (p.klen != nullptr) key_end = min(max(p.klen[bh / p.H], 0), p.N);
  // With the causal mask, Q tiles before the diagonal one (BQ == BK) see none
  // of these keys; nq counts the Q tiles visited, from q_first on.
  const int q_first = p.causal ? kv0 / C::BQ : 0;
  const int nq = kv0 < key_end ? (p.N + C::BQ - 1) / C::BQ - q_first : 0;
  if (nq == 0) {
    // Every key of this tile is masked: its dK and dV rows are zero and it
    // adds nothing to dQ. Nothing has been set up yet.
    const int rows = min(C::BK, p.N - kv0);
    const long long first = (static_cast<long long>(bh) * p.N + kv0) * D;  // 16-bit elements
    const int n16 = rows * D / 8;                                          // 16-byte chunks
    uint4* dk = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dk) + first);
    uint4* dv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dv) + first);
    for (int x = threadIdx.x; x < n16; x += C::THREADS) {
      dk[x] = make_uint4(0u, 0u, 0u, 0u);
      dv[x] = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(bbar<D>(base, C::B_K), 1);
    mbar_init(bbar<D>(base, C::B_V), 1);
    for (int s = 0; s < C::QST; ++s) {
      mbar_init(bbar<D>(base, C::B_QF + s), 1);
      mbar_init(bbar<D>(base, C::B_QE + s), 1);
    }
    for (int s = 0; s < C::OST; ++s) {
      mbar_init(bbar<D>(base, C::B_OF + s), 1);
      mbar_init(bbar<D>(base, C::B_OE + s), 1);
    }
    mbar_init(bbar<D>(base, C::B_SF), 1);
    mbar_init(bbar<D>(base, C::B_DPF), 1);
    mbar_init(bbar<D>(base, C::B_PF), 8);   // one arrival per softmax warp
    mbar_init(bbar<D>(base, C::B_DSF), 8);
    mbar_init(bbar<D>(base, C::B_DQF), 1);
    mbar_init(bbar<D>(base, C::B_DQE), 4);  // one arrival per dQ warp
    mbar_init(bbar<D>(base, C::B_DSE), 1);
    mbar_init(bbar<D>(base, C::B_DONE), 2);  // one commit per MMA warp
    misc[1] = 0;
    mbar_init_fence();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(base + C::OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const BCtl ctl{p, base + C::OFF_MISC + 4};
  if (threadIdx.x == 0) FA_TRACE(p, kBvCta, 0);

  if (warp >= 12) {
    warpgroup_reg_dealloc<C::LOW_REGS>();
    if (warp == C::WARP_TMA) {
      if ((threadIdx.x & 31) == 0) bwd_producer<D>(p, base, bh, kv0, q_first, nq, ctl);
      __syncwarp();
    } else if (warp == C::WARP_MMA) {
      bwd_mma_dsdep<D, BF16>(p, base, tmem, nq, ctl);
      __syncwarp();
    } else if (warp == C::WARP_MMA_SP) {
      bwd_mma_sp<D, BF16>(p, base, tmem, nq, ctl);
      __syncwarp();
    }
  } else if (warp >= 8) {
    warpgroup_reg_alloc<C::DQ_REGS>();
    bwd_dq<D>(p, base, tmem, bh, q_first, nq, ctl);
  } else if (warp >= 4) {
    warpgroup_reg_alloc<C::SM_REGS>();
    bwd_softmax<D, BF16, 1, FULL>(p, smem_raw, base, tmem, bh, kv0, nq, key_end, ctl);
  } else {
    warpgroup_reg_alloc<C::SM_REGS>();
    bwd_softmax<D, BF16, 0, FULL>(p, smem_raw, base, tmem, bh, kv0, nq, key_end, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) FA_TRACE(p, kBvCta, 1);
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// --------------------------------------------------------------------------
// Row statistics and the dQ accumulator
// --------------------------------------------------------------------------
// G = D/8 threads per row, 8 elements (16 bytes) each.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __grid_constant__ BwdParams p) {
  constexpr int G = D / 8;
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long prow = gt / G;  // padded row index: bh * n_pad + r
  const int g = static_cast<int>(gt % G);
  const long long rows = static_cast<long long>(p.B) * p.H * p.n_pad;
  // Every thread stays to the shuffle below (full warps); rows past the end do nothing.
  const bool in_range = prow < rows;
  const long long bh = in_range ? prow / p.n_pad : 0;
  const int r = in_range ? static_cast<int>(prow % p.n_pad) : 0;
  float acc = 0.f;
  const bool real = in_range && r < p.N;
  if (real) {
    const long long e = (bh * p.N + r) * D + g * 8;
    const uint4 o4 = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + e);
    const uint4 d4 = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + e);
    const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w}, dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float o0, o1, d0, d1;
      if constexpr (BF16) {
        o0 = __uint_as_float(ow[u] << 16);
        o1 = __uint_as_float(ow[u] & 0xFFFF0000u);
        d0 = __uint_as_float(dw[u] << 16);
        d1 = __uint_as_float(dw[u] & 0xFFFF0000u);
      } else {
        o0 = __half2float(__ushort_as_half(static_cast<unsigned short>(ow[u] & 0xFFFFu)));
        o1 = __half2float(__ushort_as_half(static_cast<unsigned short>(ow[u] >> 16)));
        d0 = __half2float(__ushort_as_half(static_cast<unsigned short>(dw[u] & 0xFFFFu)));
        d1 = __half2float(__ushort_as_half(static_cast<unsigned short>(dw[u] >> 16)));
      }
      acc = fmaf(o0, d0, acc);
      acc = fmaf(o1, d1, acc);
    }
    float4* z = reinterpret_cast<float4*>(p.dq_acc + e);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
  if (in_range && g == 0) {
    p.dsum[prow] = real ? acc : 0.f;
    // A row with no key to see (LSE = -inf, O = 0) gets +inf as well: P = 0, dQ = 0.
    const float l = real ? p.lse[bh * p.N + r] : -INFINITY;
    p.lse2[prow] = l > -INFINITY ? l * kLog2eB : INFINITY;
  }
}

// dQ = accumulator rounded to the 16-bit type, 8 elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const __grid_constant__ BwdParams p) {
  const long long n8 = static_cast<long long>(p.B) * p.H * p.N * p.d / 8;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4* src = reinterpret_cast<const float4*>(p.dq_acc) + 2 * i;
  const float4 a = src[0], b = src[1];
  uint4 out;
  out.x = pack2<BF16>(a.x, a.y);
  out.y = pack2<BF16>(a.z, a.w);
  out.z = pack2<BF16>(b.x, b.y);
  out.w = pack2<BF16>(b.z, b.w);
  reinterpret_cast<uint4*>(p.dq)[i] = out;
}

template <int D, bool BF16>
cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t stream) {
  using C = BCfg<D>;
  // Two instantiations: no entry masked (only the unmasked P loop compiled), or not.
  const bool full = !p.causal && p.klen == nullptr && p.N % C::BK == 0;
  auto kern = full ? fa_bwd_main_kernel<D, BF16, true> : fa_bwd_main_kernel<D, BF16, false>;
  static std::atomic<uint64_t> attr_done[2] = {0, 0};  // one bit per device ordinal (< 64)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done[full].load() & bit)) {
    // The warpgroup register split draws on the registers the CTA is launched
    // with: it is only valid at exactly LAUNCH_REGS per thread; refuse otherwise.
    cudaFuncAttributes fa_attr;
    e = cudaFuncGetAttributes(&fa_attr, kern);
    if (e != cudaSuccess) return e;
    if (fa_attr.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[full].fetch_or(bit);
  }
  const long long bh = static_cast<long long>(p.B) * p.H;
  const long long nt = (p.N + C::BK - 1) / C::BK;
  const long long pre_threads = bh * p.n_pad * (D / 8);
  const long long post_threads = bh * p.N * D / 8;
  if (bh * nt > 0x7fffffffLL || (pre_threads + 255) / 256 > 0x7fffffffLL || (post_threads + 255) / 256 > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  fa_bwd_pre_kernel<D, BF16><<<dim3(static_cast<unsigned>((pre_threads + 255) / 256)), dim3(256), 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kern<<<dim3(static_cast<unsigned>(bh * nt)), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_post_kernel<BF16><<<dim3(static_cast<unsigned>((post_threads + 255) / 256)), dim3(256), 0, stream>>>(p);
  return cudaGetLastError();
}

// d = 256: the same row statistics and dQ rounding around the two main
// kernels of fa_bwd_d256.cu.
template <bool BF16>
cudaError_t launch_bwd_d256_t(const BwdParams& p, cudaStream_t stream) {
  const long long bh = static_cast<long long>(p.B) * p.H;
  const long long pre_threads = bh * p.n_pad * (256 / 8);
  const long long post_threads = bh * p.N * 256 / 8;
  if ((pre_threads + 255) / 256 > 0x7fffffffLL || (post_threads + 255) / 256 > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  fa_bwd_pre_kernel<256, BF16><<<dim3(static_cast<unsigned>((pre_threads + 255) / 256)), dim3(256), 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_bwd_main_d256(p, BF16, stream);
  if (e != cudaSuccess) return e;
  fa_bwd_post_kernel<BF16><<<dim3(static_cast<unsigned>((post_threads + 255) / 256)), dim3(256), 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_f16(const BwdParams& p, bool bf16, cudaStream_t stream) {
  if (p.d == 256) return bf16 ? launch_bwd_d256_t<true>(p, stream) : launch_bwd_d256_t<false>(p, stream);
  if (p.d == 128) return bf16 ? launch_bwd_t<128, true>(p, stream) : launch_bwd_t<128, false>(p, stream);
  if (p.d == 64) return bf16 ? launch_bwd_t<64, true>(p, stream) : launch_bwd_t<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
