// fa_fwd_f16.cu — FlashAttention forward for fp16 / bf16 on sm_103a.
//
// Algorithm: the tiled online-softmax recurrence of the MUSA SDK guide
// ("FlashAttention 优化", "FlashAttention 完整算法", formula steps 1-4 and the
// flow chart): a Q tile stays resident, K/V tiles stream past it, for each
// tile S = Q K^T, the running row max m and denominator l are updated, O is
// rescaled by exp(m_old - m_new) before the new P V is added (the dataflow
// page, section 2.3, stresses that order), and O is divided by l at the end.
// The loop order (Q outer, K/V inner, Q loaded once) is the dataflow page's
// section 2.2; the parallelisation over Q tiles is the guide's FlashAttention-2
// "sequence parallelism" note; overlapping the next tile's Q K^T with the
// current tile's softmax is the guide's FlashAttention-3 pipelining note.
//
// GB300 mapping (one CTA per (batch*head, 256-row Q block), 12 warps):
//   warp 9      TMA producer: Q0/Q1 once, then K_j and V_j (128 keys each)
//               into 2-stage (d=128) / 3-stage (d=64) rings; for d=128 the
//               softmax warps free a stage once the S product they wait for
//               shows that its K (and the previous tile's V) have been read,
//               for d=64 commits behind the MMAs do
//   warps 8, 10 MMA warps, one per Q sub-tile i (d=128; at d=64 warp 8
//               issues for both): S_i(j) = Q_i K_j^T (SS, into TMEM), then
//               O_i += P_i(j) V_j (TS: P read from TMEM, V from SMEM); one
//               elected lane issues; warp 8 also owns TMEM
//   warps 0-3   softmax for Q rows 0-127   (thread = row; TMEM lanes = rows)
//   warps 4-7   softmax for Q rows 128-255
//   warp 11     idle (completes the third warpgroup for the register split)
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [256+d,256+2d).
// P_i(j) (16-bit, packed in pairs) overwrites the first 64 columns of S_i.
// S_i(j+1) is issued right behind P_i(j) V_j by the same warp: the M=128 MMA
// occupies the whole SM tensor core and one CTA's MMAs execute in issue order,
// so S_i(j+1) cannot overwrite P_i(j) before it is read (the PTX ISA states
// this ordering only for MMAs on the same accumulator; building with
// -DFA_STRICT_MMA_ORDER waits for P_i(j) V_j to complete instead).
// One MMA warp per sub-tile drives the chain S_i -> softmax_i -> P_i V -> S_i;
// the two warps pass a turn so that their MMA blocks alternate (ping-pong) and
// each runs inside the other chain's softmax (d=64: one warp issues the blocks
// of both chains in that order).
// Each tile's row max comes with the TMEM load of its scores (sm_103a's
// tcgen05.ld with a max reduction), so no max tree over the scores stands
// between the load and the exponentials; tiles with masked keys take the max
// in registers after masking. The rescale of O is lazy: the reference max
// only moves when the tile max exceeds it by more than the threshold (15 in
// log2 units), so P <= 2^15 and rescales are rare.
// The epilogue divides by l, rounds to the input type, stages the tile in the
// (now unused) Q buffer in the TMA 128-byte swizzle layout and TMA-stores it;
// LSE = ln2 * (m + log2 l) is written per row.
#include <atomic>

#include "fa_device_common.cuh"
#include "fa_fwd_order.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
#ifdef FA_STRICT_MMA_ORDER
constexpr bool kOdEveryTile = true;   // every P.V committed to o_done (S waits for it)
#else
constexpr bool kOdEveryTile = false;  // only the last P.V of a sub-tile
#endif

template <int D>
struct Cfg {
  static constexpr int BM = kF16BlockQ;   // Q rows per sub-tile (= TMEM lanes)
  static constexpr int BN = kF16BlockKV;  // keys per K/V tile
  static constexpr int STAGES = (D == 128) ? 2 : 3;
  // Who frees the K/V stages: the softmax warps (d = 128: keeps commits out
  // of the MMA issue stream, whose blocks are long) or commits behind the MMAs
  // (d = 64: short blocks, and the softmax is the longer part of the chain).
  static constexpr bool SOFTMAX_FREES_STAGES = (D == 128);
  static constexpr uint32_t ROW_BYTES = 128;               // one 128-byte swizzle row = 64 elements
  static constexpr uint32_t Q_SUB_BYTES = BM * D * 2;      // one Q sub-tile
  static constexpr uint32_t Q_HALF_BYTES = BM * ROW_BYTES; // 64 columns of a Q sub-tile
  static constexpr uint32_t KV_BYTES = BN * D * 2;         // one K or V tile
  static constexpr uint32_t KV_HALF_BYTES = BN * ROW_BYTES;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * Q_SUB_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
  // barriers: q | k_full[S] | k_empty[S] | v_full[S] | v_empty[S] |
  //           s_full[2] | p_full[2] | o_done[2] | drain[2] | turn[2]     ([sub])
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;
  static constexpr int B_KE = B_KF + STAGES;
  static constexpr int B_VF = B_KE + STAGES;
  static constexpr int B_VE = B_VF + STAGES;
  static constexpr int B_SF = B_VE + STAGES;
  static constexpr int B_PF = B_SF + 2;
  static constexpr int B_OD = B_PF + 2;
  static constexpr int B_DRAIN = B_OD + 2;
  static constexpr int B_TURN = B_DRAIN + 2;
  static constexpr int NBAR = B_TURN + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_O0 = 256, T_O1 = 256 + D;
  // 3 warpgroups: softmax sub-tile 0, softmax sub-tile 1, and {MMA 0, TMA, MMA 1, idle} warps.
  static constexpr int THREADS = 384;
  static constexpr int WARP_MMA0 = 8, WARP_TMA = 9, WARP_MMA1 = 10;
  // Register split: launched at LAUNCH_REGS per thread (the compiler's count for
  // 384 threads, checked on the host before launch), the producer/MMA
  // warpgroup gives back down to LOW_REGS and each softmax warpgroup grows to
  // HIGH_REGS: 2*128*HIGH + 128*LOW <= 384*LAUNCH.
  static constexpr int LAUNCH_REGS = 168, HIGH_REGS = 216, LOW_REGS = 72;
  static_assert(2 * 128 * HIGH_REGS + 128 * LOW_REGS <= THREADS * LAUNCH_REGS, "register split exceeds the pool");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// TMEM column of S_i (and of P_i, which overwrites its first 64 columns).
__device__ __forceinline__ uint32_t t_s_col(int sub) { return 128u * sub; }

template <int D>
__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) {
  return base + Cfg<D>::OFF_BAR + 8u * i;
}

// --------------------------------------------------------------------------
// TMA producer (one thread)
// --------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void producer(const FwdParams& p, uint32_t base, int bh, int row0, bool has1, int t0,
                                         int nkv, const WaitCtl& ctl) {
  using C = Cfg<D>;
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);
  tma_prefetch_desc(&p.tm_o);

  // A unit with no key tile (key length 0) loads nothing: its epilogue writes
  // zeros into the Q buffers, which no copy may land in afterwards.
  if (nkv == 0) return;
  const uint32_t bq = bar_addr<D>(base, C::B_Q);
  mbar_arrive_expect_tx(bq, (has1 ? 2u : 1u) * C::Q_SUB_BYTES);
  for (int sub = 0; sub < (has1 ? 2 : 1); ++sub)
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_load_3d(base + C::OFF_Q + sub * C::Q_SUB_BYTES + h * C::Q_HALF_BYTES, &p.tm_q, bq, 64 * h,
                  row0 + C::BM * sub, bh);

  int nk = 0, nv = 0;  // K / V tiles whose loads were issued
  bool ok = true;
  for (int j = 0; j < nkv; ++j) {
    const int s = j % C::STAGES;
    const uint32_t par = ((j / C::STAGES) & 1) ^ 1;
    if (!wait_bar(bar_addr<D>(base, C::B_KE + s), par, ctl, kWhereKEmpty)) { ok = false; break; }
    const uint32_t kf = bar_addr<D>(base, C::B_KF + s);
    mbar_arrive_expect_tx(kf, C::KV_BYTES);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_load_3d(base + C::OFF_K + s * C::KV_BYTES + h * C::KV_HALF_BYTES, &p.tm_k, kf, 64 * h, (t0 + j) * C::BN, bh);
    nk = j + 1;
    FA_TRACE(p, kEvKIssued, j);
#ifdef FA_TESTING
    if (p.inject == 1 && j == 0) continue;  // fault injection: V_0 is never loaded
#endif
    if (!wait_bar(bar_addr<D>(base, C::B_VE + s), par, ctl, kWhereVEmpty)) { ok = false; break; }
    const uint32_t vf = bar_addr<D>(base, C::B_VF + s);
    mbar_arrive_expect_tx(vf, C::KV_BYTES);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_load_3d(base + C::OFF_V + s * C::KV_BYTES + h * C::KV_HALF_BYTES, &p.tm_v, vf, 64 * h, (t0 + j) * C::BN, bh);
    nv = j + 1;
    FA_TRACE(p, kEvVIssued, j);
  }
  // Drain: every copy this thread started must land before the CTA exits,
  // whether the loop ended normally, this thread's own wait gave up, or
  // another role aborts later (its waits give up only after the last loads
  // were issued). The most recent load of each stage is one of the last
  // STAGES tiles issued. Cheap when nothing failed: the consumers need these
  // copies anyway, so they land before the CTA could finish.
  (void)ok;
  {
    wait_bar_drain(bq, 0, ctl);
    for (int t = nk > C::STAGES ? nk - C::STAGES : 0; t < nk; ++t)
      wait_bar_drain(bar_addr<D>(base, C::B_KF + t % C::STAGES), (t / C::STAGES) & 1, ctl);
    for (int t = nv > C::STAGES ? nv - C::STAGES : 0; t < nv; ++t) {
#ifdef FA_TESTING
      if (p.inject == 1 && t == 0) continue;  // never armed
#endif
      wait_bar_drain(bar_addr<D>(base, C::B_VF + t % C::STAGES), (t / C::STAGES) & 1, ctl);
    }
  }
}

// --------------------------------------------------------------------------
// MMA issue (whole warp; one elected lane issues)
// --------------------------------------------------------------------------
// Block j of sub-tile SUB's chain: P(j-1) V_{j-1}, then S(j) = Q K_j^T.
// gkv is the position of tile j in the CTA's sequence of K/V tiles (its ring
// stage and phase), gp the position of P(j) in the sub-tile's sequence of P
// tiles (equal to j for a CTA with one work unit). Returns false when a wait
// gave up.
template <int D, bool BF16, int SUB>
__device__ __forceinline__ bool mma_block(const FwdParams& p, uint32_t base, uint32_t tmem, int j, int nkv, int gkv,
                                          int gp, const WaitCtl& ctl) {
  using C = Cfg<D>;
  constexpr int sub = SUB;
  constexpr uint32_t fmt = BF16 ? 1u : 0u;
  // S = Q K^T: A = Q (K-major), B = K tile (K-major), M = 128, N = 128.
  constexpr uint32_t idesc_qk = make_idesc(fmt, 0, 0, 128, C::BN);
  // O += P V: A = P from TMEM (K-major), B = V tile, N (= d) contiguous -> MN-major.
  constexpr uint32_t idesc_pv = make_idesc(fmt, 0, 1, 128, D);
  // 16 keys = two 8-row swizzle atoms (SBO apart); the two 64-wide halves of d are LBO apart.
  // With d = 64 there is one half and LBO is unused; 1024 keeps every address inside the tile.
  constexpr uint32_t lbo = (D == 64) ? 1024u : C::KV_HALF_BYTES;
  const uint32_t d_s = tmem + t_s_col(sub);
  const uint32_t d_o = tmem + (sub ? C::T_O1 : C::T_O0);
  const uint32_t qbase = base + C::OFF_Q + sub * C::Q_SUB_BYTES;
  const uint32_t b_sf = bar_addr<D>(base, C::B_SF + sub), b_pf = bar_addr<D>(base, C::B_PF + sub);
  const uint32_t b_od = bar_addr<D>(base, C::B_OD + sub);
  if (j > 0) {
    // P(j-1) V_{j-1}
    const int s = (gkv - 1) % C::STAGES;
    if (!wait_bar_warp(bar_addr<D>(base, C::B_VF + s), ((gkv - 1) / C::STAGES) & 1, ctl, kWhereVFull)) return false;
    if (!wait_bar_warp(b_pf, (gp - 1) & 1, ctl, kWherePFull)) return false;
    tc_fence_after();
    if (sub == 0) FA_TRACE(p, kEvMmaVFull, j - 1);
    const uint64_t v0 = smem_desc_sw128(base + C::OFF_V + s * C::KV_BYTES, lbo, 1024);
#pragma unroll
    for (int kk = 0; kk < C::BN / 16; ++kk)
      mma_f16_ts_elect(d_o, d_s + kk * 8, v0 + ((kk * 16 * C::ROW_BYTES) >> 4), idesc_pv,
                       (j > 1 || kk > 0) ? 1u : 0u);
    // The softmax learns that P(j-1) V_{j-1} is complete from the commit that
    // follows S(j) (same warp, issued after it); only the last P.V, which no
    // S follows, is committed on its own (strict order: every P.V is).
    if (kOdEveryTile || j == nkv) tc_commit_elect(b_od);
    if constexpr (!C::SOFTMAX_FREES_STAGES) tc_commit_elect(bar_addr<D>(base, C::B_VE + s));
    FA_TRACE(p, kEvPV0Issued + sub, j - 1);
  }
  if (j < nkv) {
    // S(j) = Q K_j^T. P(j-1) lives in the S columns: S(j) must not overwrite
    // them before P(j-1) V_{j-1} has read them. By default S(j) is issued right
    // behind that P.V (same warp, same tensor pipe, executed in issue order);
    // FA_STRICT_MMA_ORDER waits for the P.V to complete first.
    const int s = gkv % C::STAGES;
    if (!wait_bar_warp(bar_addr<D>(base, C::B_KF + s), (gkv / C::STAGES) & 1, ctl, kWhereKFull)) return false;
#ifdef FA_STRICT_MMA_ORDER
    if (j > 0 && !wait_bar_warp(b_od, (j - 1) & 1, ctl, kWhereODone)) return false;
#endif
    tc_fence_after();
    if (sub == 0) FA_TRACE(p, kEvMmaKFull, j);
    // Descriptors of k-step 0; later k-steps advance the 14-bit start-address
    // field (bytes >> 4), which cannot carry out since shared addresses < 2^18.
    const uint64_t a0 = smem_desc_sw128(qbase, 16, 1024);
    const uint64_t b0 = smem_desc_sw128(base + C::OFF_K + s * C::KV_BYTES, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      // 16 elements = 32 bytes inside the swizzled row; every 4 k-steps the next 64-column half
      const uint32_t aoff = ((kk / 4) * C::Q_HALF_BYTES + (kk & 3) * 32u) >> 4;
      const uint32_t boff = ((kk / 4) * C::KV_HALF_BYTES + (kk & 3) * 32u) >> 4;
      mma_f16_ss_elect(d_s, a0 + aoff, b0 + boff, idesc_qk, kk > 0 ? 1u : 0u);
    }
    tc_commit_elect(b_sf);
    if constexpr (!C::SOFTMAX_FREES_STAGES) tc_commit_elect(bar_addr<D>(base, C::B_KE + s));
    FA_TRACE(p, kEvS0Issued + sub, j);
  }
  return true;
}

// d = 128: one MMA warp per Q sub-tile. Chain i alternates on the tensor pipe
// with the other sub-tile's chain in blocks B_i(j) = { P_i(j-1) V_{j-1} ;
// S_i(j) = Q_i K_j^T }, in the order B_0(0), B_1(0), B_0(1), B_1(1), ... A warp
// passes the turn (an mbarrier arrival) after issuing its block. Between its
// blocks each chain runs its softmax, so one chain's block executes inside the
// other chain's softmax window instead of both chains requesting the pipe at
// the same time.
template <int D, bool BF16, int SUB>
__device__ __forceinline__ void mma_warp(const FwdParams& p, uint32_t base, uint32_t tmem, bool has1, int nkv,
                                         int nkv_other, const WaitCtl& ctl) {
  using C = Cfg<D>;
  constexpr int sub = SUB;
  const uint32_t b_drain = bar_addr<D>(base, C::B_DRAIN + sub);
  const uint32_t my_turn = bar_addr<D>(base, C::B_TURN + sub), next_turn = bar_addr<D>(base, C::B_TURN + (sub ^ 1));

  if (nkv == 0) goto drain;  // no key to attend to (key length 0): nothing to issue
  if (!wait_bar_warp(bar_addr<D>(base, C::B_Q), 0, ctl, kWhereQ)) goto drain;
  tc_fence_after();
  for (int j = 0; j <= nkv; ++j) {
    // My block j follows the other chain's block j-1 (sub 0) or block j (sub 1),
    // as long as the other chain has that block (its tile count can differ).
    const int other = sub == 1 ? j : j - 1;
    if (has1 && other >= 0 && other <= nkv_other && nkv_other > 0) {
      if (!wait_bar_warp(my_turn, other & 1, ctl, kWhereTurn)) goto drain;
    }
    if (!mma_block<D, BF16, SUB>(p, base, tmem, j, nkv, j, j, ctl)) goto drain;
    if (has1) {
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(next_turn);
    }
  }
drain:
  // All MMAs issued by this warp complete before the CTA may free TMEM / exit.
  tc_commit_elect(b_drain);
  __all_sync(0xffffffffu, wait_bar_drain(b_drain, 0, ctl));
}

// d = 64: one MMA warp issues both chains' blocks in the same order
// (B_0(0), B_1(0), B_0(1), ...) by program order instead of turns: the blocks
// are short there and the turn handoff between two warps cost more than the
// second warp's overlap of waits and commits gained.
template <int D, bool BF16>
__device__ __forceinline__ void mma_both(const FwdParams& p, uint32_t base, uint32_t tmem, bool has1, int nkv0,
                                         int nkv1, const WaitCtl& ctl) {
  const uint32_t b_drain = bar_addr<D>(base, Cfg<D>::B_DRAIN);
  const int n = max(nkv0, nkv1);
  if (n > 0 && wait_bar_warp(bar_addr<D>(base, Cfg<D>::B_Q), 0, ctl, kWhereQ)) {
    tc_fence_after();
    for (int j = 0; j <= n; ++j) {
      if (nkv0 > 0 && j <= nkv0 && !mma_block<D, BF16, 0>(p, base, tmem, j, nkv0, j, j, ctl)) break;
      if (has1 && nkv1 > 0 && j <= nkv1 && !mma_block<D, BF16, 1>(p, base, tmem, j, nkv1, j, j, ctl)) break;
    }
  }
  // All MMAs issued by this warp complete before the CTA may free TMEM / exit.
  tc_commit_elect(b_drain);
  __all_sync(0xffffffffu, wait_bar_drain(b_drain, 0, ctl));
}

// One key tile of a sub-tile's softmax: wait for S(j), release the K/V
// stages it shows read, take the tile's row max, decide the lazy rescale,
// write P over the S columns, rescale O when decided, and hand P to the MMA
// warp. valid: keys of this tile the row may see; gkv: position of tile j in
// the CTA's K/V ring sequence; gs: position of S(j) in the sub-tile's
// sequence of S products (both equal to j for a CTA with one work unit).
// Returns false when a wait gave up.
template <int D, bool BF16>
__device__ __forceinline__ bool softmax_tile(const FwdParams& p, uint32_t base, int sub, int t, int lane,
                                             uint32_t t_s, uint32_t t_o, float c, float tau, int valid, int j,
                                             int gkv, int gs, float& m_ref, float& l, float& l_o,
                                             const WaitCtl& ctl) {
  using C = Cfg<D>;
  (void)p;
  const uint32_t b_sf = bar_addr<D>(base, C::B_SF + sub), b_pf = bar_addr<D>(base, C::B_PF + sub);
  const uint32_t b_od = bar_addr<D>(base, C::B_OD + sub);
  (void)b_od;
  // Wait results are made warp-uniform: TMEM loads/stores below need the whole warp.
  if (!__all_sync(0xffffffffu, wait_bar(b_sf, gs & 1, ctl, kWhereSFull))) return false;
  tc_fence_after();
  if (t == 0) FA_TRACE(p, kEvSm0SFull + 2 * sub, j);
  if (C::SOFTMAX_FREES_STAGES && lane == 0) {
    // The K/V stages are released from here, not by commits in the MMA
    // warp's issue stream (a commit right behind a group of MMAs leaves the
    // tensor pipe idle for ~200 cycles): S(j) is complete, so K_j has been
    // read, and so has V_{j-1}, since P(j-1) V_{j-1} was issued before S(j)
    // by the same warp and one commit covers all of its earlier MMAs.
    // V first: once the producer sees a K phase complete, every warp's
    // earlier V arrival has happened, so no warp can arrive for a stage's
    // next tile while its current phase is still open.
    if (j > 0) mbar_arrive(bar_addr<D>(base, C::B_VE + (gkv - 1) % C::STAGES));
    mbar_arrive(bar_addr<D>(base, C::B_KE + gkv % C::STAGES));
  }
  // S in registers, with each 32-column block's row max from the same load
  // (the TMEM load with a max reduction of sm_103a).
  uint32_t sraw[C::BN / 32][32];
  float mxq[C::BN / 32];
#pragma unroll
  for (int q = 0; q < C::BN / 32; ++q) tmem_ld32_max(t_s + 32 * q, sraw[q], mxq[q]);
  tmem_ld_wait();
  float s[C::BN];
#pragma unroll
  for (int q = 0; q < C::BN / 32; ++q) {
    reg_fence(sraw[q]);
    asm volatile("" : "+f"(mxq[q]));  // valid only after the wait, like sraw
#pragma unroll
    for (int u = 0; u < 32; ++u) s[32 * q + u] = __uint_as_float(sraw[q][u]);
  }

  float mx = mxq[0];
#pragma unroll
  for (int q = 1; q < C::BN / 32; ++q) mx = fmaxf(mx, mxq[q]);
  if (valid < C::BN) {
    // Masked keys (the ragged end, the diagonal, a key length) become -inf
    // and the max is taken over the rest: the loads' max includes them.
#pragma unroll
    for (int u = 0; u < C::BN; ++u)
      if (u >= valid) s[u] = -INFINITY;
    float mxa[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mxa[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
    for (int u = 16; u < C::BN; u += 16)
#pragma unroll
      for (int i = 0; i < 8; ++i) mxa[i] = fmax3(mxa[i], s[u + i], s[u + 8 + i]);
    mx = fmaxf(fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])), fmaxf(fmaxf(mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7])));
  }
  const float m_new = fmaxf(m_ref, mx * c);

  // Lazy rescale decision (warp-uniform, since TMEM access is per warp): move
  // the reference max of every row of this warp when any row's tile max
  // exceeds it by more than the threshold. l is rescaled now; O is rescaled
  // below, after P is stored but before P is released to the P.V MMA.
  bool rescale_o = false;
  float alpha = 1.f;
  if (j == 0) {
    m_ref = m_new;  // O is written fresh by the first P.V; l is 0
  } else if (__any_sync(0xffffffffu, m_new - m_ref > tau)) {
    // = exp(m_old - m_new) in natural units; 0 for a row that saw no key
    // yet (its l and O are 0), never exp2(-inf + inf)
    alpha = m_ref > -INFINITY ? ex2_approx(m_ref - m_new) : 0.f;
    m_ref = m_new;
    l *= alpha;
    l_o *= alpha;
    rescale_o = true;
  }

  // P = 2^(s*c - m_ref), two scores per packed FMA. The exact fp32 sum gives
  // l (for LSE). For bf16 the P.V product sees P rounded to 8 significant
  // bits, so O is normalised by the sum of the rounded P (l_o): numerator
  // and denominator then use the same weights, which keeps |dO| well below
  // the rounding of a bf16 output even for sharply peaked rows.
  // A row that has seen no key yet (every score so far masked: possible in
  // a key range of a split under the causal mask) keeps m_ref = -inf; its
  // P are computed against 0 so that they are 0, not exp2(-inf + inf).
  const float m_use = m_ref > -INFINITY ? m_ref : 0.f;
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(-m_use, -m_use);
  float2 se = make_float2(0.f, 0.f), sro = se;  // exact / rounded partial sums
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
        // fp32 adds (exact conversion, one add each): cheaper than
        // unpacking them into fp32 registers first.
        unsigned short lo16, hi16;
        asm("mov.b32 {%0, %1}, %2;" : "=h"(lo16), "=h"(hi16) : "r"(pk[u]));
        asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(sro.x) : "h"(lo16));
        asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(sro.y) : "h"(hi16));
      }
    }
    tmem_st8(t_s + 8 * q, pk);  // keys [16q, 16q+16) -> packed columns [8q, 8q+8)
  }
  l += se.x + se.y;
  if constexpr (BF16) l_o += sro.x + sro.y;
  if (rescale_o) {
    // O must be complete up to tile j-1 (its P.V finished) before it is read
    // and scaled. P(j-1) V_{j-1} was issued before S(j) by the same warp, so
    // the S(j) completion waited for above covers it; the strict build
    // commits and waits for every P.V.
    if (kOdEveryTile && !__all_sync(0xffffffffu, wait_bar(b_od, (gs - 1) & 1, ctl, kWhereODone))) return false;
    tc_fence_after();
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
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
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(b_pf);
  if (t == 0) FA_TRACE(p, kEvSm0PArrive + 2 * sub, j);
  return true;
}

// --------------------------------------------------------------------------
// Softmax + lazy correction + epilogue (one warpgroup per Q sub-tile)
// --------------------------------------------------------------------------
// FULL: no key of any tile is masked (no causal mask, no key lengths, a
// multiple of 128 keys), so the masked path of the tile is compiled out.
template <int D, bool BF16, bool FULL>
__device__ __forceinline__ void softmax_wg(const FwdParams& p, uint32_t base, uint32_t tmem, int sub, int bh, int row0,
                                           int split, int t0, int nkv, int key_end, const WaitCtl& ctl) {
  using C = Cfg<D>;
  const int t = threadIdx.x - sub * 128;  // row within the sub-tile
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = static_cast<uint32_t>(t & ~31) << 16;
  const uint32_t t_o = tmem + lane_base + (sub ? C::T_O1 : C::T_O0);
  const float c = p.scale * kLog2e;  // scores in log2 units: x = s * c
  // Keys this row may see: [0, row_end) (all keys up to key_end; causal: up to the row itself).
  const int my_row = row0 + C::BM * sub + t;
  const int row_end = p.causal ? min(key_end, my_row + 1) : key_end;

  const float tau = rescale_threshold(p);
  float m_ref = -INFINITY;  // reference max (log2 units) shared by l and O
  float l = 0.f;            // sum of P (fp32) relative to m_ref: gives LSE
  float l_o = 0.f;          // bf16 only: sum of the rounded P: normalises O
  bool ok = true;

  const uint32_t t_s = tmem + lane_base + t_s_col(sub);
  const uint32_t b_od = bar_addr<D>(base, C::B_OD + sub);

  for (int j = 0; j < nkv; ++j) {
    const int valid = FULL ? C::BN : row_end - (t0 + j) * C::BN;
    if (!softmax_tile<D, BF16>(p, base, sub, t, lane, t_s, t_o, c, tau, valid, j, j, j, m_ref, l, l_o, ctl)) {
      ok = false;
      break;
    }
#ifdef FA_TESTING
    if (p.stats_trace) {
      const int row = row0 + C::BM * sub + t;
      if (row < p.N) {
        float* tr = p.stats_trace + ((static_cast<size_t>(bh) * p.N + row) * nkv + j) * 2;
        tr[0] = m_ref * kLn2;
        tr[1] = l;
      }
    }
#endif
  }
  // The last P.V of this sub-tile; its commit also covers every earlier MMA of the warp.
  if (ok && nkv > 0)
    ok = __all_sync(0xffffffffu, wait_bar(b_od, kOdEveryTile ? (nkv - 1) & 1 : 0, ctl, kWhereODone));
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
    // normalised O (fp32) and LSE go to the partial buffers.
    const int row = row0 + C::BM * sub + t;
    // Partial rows are numbered from merge_row0 (the first row of the split
    // units; 0 unless only the wave tail is split), one span per key range.
    const size_t span = static_cast<size_t>(p.B) * p.H * p.N - p.merge_row0;
    const size_t prow = static_cast<size_t>(split) * span + (static_cast<size_t>(bh) * p.N + row - p.merge_row0);
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
      uint32_t r[32];
      tmem_ld32(t_o + 32 * q, r);
      tmem_ld_wait();
      reg_fence(r);
      if (empty) {
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] = 0u;  // no key in this range: O_part = 0, LSE_part = -inf
      }
      if (row < p.N) {
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D + 32 * q);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          dst[u] = make_float4(__uint_as_float(r[4 * u]) * inv_l, __uint_as_float(r[4 * u + 1]) * inv_l,
                               __uint_as_float(r[4 * u + 2]) * inv_l, __uint_as_float(r[4 * u + 3]) * inv_l);
      }
    }
    if (row < p.N) p.lse_part[prow] = empty ? -INFINITY : (m_ref + lg2_approx(l)) * kLn2;
    return;
  }
  const uint32_t stage = base + C::OFF_Q + sub * C::Q_SUB_BYTES;
#pragma unroll
  for (int q = 0; q < D / 32; ++q) {
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
      const uint32_t addr = stage + half * C::Q_HALF_BYTES + t * C::ROW_BYTES + phys * 16;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * u]), "r"(pk[4 * u + 1]),
                   "r"(pk[4 * u + 2]), "r"(pk[4 * u + 3])
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  named_bar_sync(1 + sub, 128);
  if (t == 0) {
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_store_3d(&p.tm_o, stage + h * C::Q_HALF_BYTES, 64 * h, row0 + C::BM * sub, bh);
    tma_store_commit();
    tma_store_wait_all();
  }
  const int row = row0 + C::BM * sub + t;
  if (row < p.N) p.lse[static_cast<size_t>(bh) * p.N + row] = empty ? -INFINITY : (m_ref + lg2_approx(l)) * kLn2;
}

template <int D, bool BF16, bool FULL>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1) fa_fwd_f16_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem_raw + (base - raw) + C::OFF_MISC);

  const int warp = threadIdx.x >> 5;
  // Work unit: (batch*head, 256-row Q block, key range), in the order of
  // fa_fwd_order.cuh: a head's Q blocks in a row; causal launches over every
  // unit unsplit, longest first within windows of heads. Split launches keep
  // the natural order, in which the units of the split-KV tail plan (the
  // last ones) hold the last rows: its merge and partial buffers cover the
  // rows from merge_row0 on.
  const int nqb = (p.N + 2 * C::BM - 1) / (2 * C::BM);
  const int split = blockIdx.x % p.num_splits;
  const int qunit = p.qunit0 + blockIdx.x / p.num_splits;
  const bool heavy_first = p.causal && p.num_splits == 1 && p.qunit_count == 0;
  const FwdUnitOf unit = fwd_unit_of(qunit, p.B * p.H, nqb, p.Nk, D, heavy_first, p.num_sms);
  const int bh = unit.bh;
  const int qb = unit.qb;
  const int row0 = qb * 2 * C::BM;
  const bool has1 = row0 + C::BM < p.N;
  // Keys this unit may see: [0, key_end); causal limits each sub-tile to its own last row.
  const int key_end = p.klen ? max(0, min(p.Nk, p.klen[bh / p.H])) : p.Nk;
  const int end0 = p.causal ? min(key_end, row0 + C::BM) : key_end;
  const int end1 = p.causal ? min(key_end, row0 + 2 * C::BM) : key_end;
  const int t0 = split * p.split_tiles;                      // first K/V tile of this key range
  // Tiles per sub-tile in this key range (none when its keys end before the range starts).
  const int nkv0 = max(0, min((end0 + C::BN - 1) / C::BN - t0, p.split_tiles));
  const int nkv1 = has1 ? max(0, min((end1 + C::BN - 1) / C::BN - t0, p.split_tiles)) : 0;
  const int nkv = max(nkv0, nkv1);                           // tiles the producer loads

  if (threadIdx.x == 0) {
    mbar_init(bar_addr<D>(base, C::B_Q), 1);
    const uint32_t nsub = has1 ? 2u : 1u;  // the stage-empty barriers get releases from each sub-tile
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_addr<D>(base, C::B_KF + s), 1);
      // one arrival per softmax warp (d = 128) or one commit per MMA warp (d = 64)
      mbar_init(bar_addr<D>(base, C::B_KE + s), C::SOFTMAX_FREES_STAGES ? 4 * nsub : nsub);
      mbar_init(bar_addr<D>(base, C::B_VF + s), 1);
      mbar_init(bar_addr<D>(base, C::B_VE + s), C::SOFTMAX_FREES_STAGES ? 4 * nsub : nsub);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_addr<D>(base, C::B_SF + i), 1);
      mbar_init(bar_addr<D>(base, C::B_PF + i), 4);  // one arrival per softmax warp
      mbar_init(bar_addr<D>(base, C::B_OD + i), 1);
      mbar_init(bar_addr<D>(base, C::B_DRAIN + i), 1);
      mbar_init(bar_addr<D>(base, C::B_TURN + i), 1);
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
  // A split tail launched behind this kernel (a programmatic dependent that
  // reads none of its results) may start its CTAs as this kernel's finish.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) FA_TRACE(p, kEvCta, 0);

  if (warp >= 8) {
    warpgroup_reg_dealloc<C::LOW_REGS>();
    if (warp == C::WARP_TMA) {
      if ((threadIdx.x & 31) == 0) producer<D>(p, base, bh, row0, has1, t0, nkv, ctl);
      __syncwarp();
    } else if (D == 64 && warp == C::WARP_MMA0) {
      mma_both<D, BF16>(p, base, tmem, has1, nkv0, nkv1, ctl);
      __syncwarp();
    } else if (D != 64 && (warp == C::WARP_MMA0 || (warp == C::WARP_MMA1 && has1))) {
      if (warp == C::WARP_MMA0)
        mma_warp<D, BF16, 0>(p, base, tmem, has1, nkv0, nkv1, ctl);
      else
        mma_warp<D, BF16, 1>(p, base, tmem, has1, nkv1, nkv0, ctl);
      __syncwarp();
    }
  } else {
    warpgroup_reg_alloc<C::HIGH_REGS>();
    const int sub = warp / 4;
    if (sub == 0 || has1)
      softmax_wg<D, BF16, FULL>(p, base, tmem, sub, bh, row0, split, t0, sub ? nkv1 : nkv0, key_end, ctl);
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
  // Launched as a programmatic dependent (the split tail after the full
  // rounds): finish only after the kernel before it (no-op otherwise).
  if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ==========================================================================
// Persistent form (d = 128, unmasked or causal, and unmasked d = 64; no
// key-range split, no key lengths, N a multiple of 256, at most 4096):
// one CTA per SM walks the work units blockIdx.x, blockIdx.x + G, ... (G
// CTAs), so a unit's Q and first K/V tiles load while the previous unit's
// last tiles and epilogue run, instead of paying a CTA's start and end per
// unit. The barriers continue their phases from unit to unit: every role
// counts the K/V tiles (ring stages and phases), S and P products and units
// it has seen. One MMA warp issues both chains' blocks in turn order. Three
// more barriers: the Q buffer is free (the last S product of both sub-tiles
// has completed), and O_i has been read out by the epilogue (the next unit's
// first P.V overwrites it). The epilogue stages O in 64-column halves through
// a 16 KB buffer of each sub-tile, since the Q buffer already holds the next
// unit's Q. Separate instantiations for unmasked, causal and streamed-tail
// launches carry only their own code (the kernels' speed depends on their
// size); the unmasked ones compile the key mask out.
// ==========================================================================
template <int D>
struct PCfg {
  using C = Cfg<D>;
  static constexpr uint32_t OFF_XBAR = C::OFF_MISC + 16;  // Q free | O0 free | O1 free
  static constexpr int X_QE = 0, X_OF = 1;
  static constexpr uint32_t OFF_STG = (OFF_XBAR + 3 * 8 + 1023u) & ~1023u;
  static constexpr uint32_t STG_BYTES = C::Q_HALF_BYTES;  // 64 columns of a 128-row sub-tile
  static constexpr uint32_t SMEM_BYTES = OFF_STG + 2 * STG_BYTES + 1024;  // + slack to align the base
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int D>
__device__ __forceinline__ uint32_t xbar_addr(uint32_t base, int i) {
  return base + PCfg<D>::OFF_XBAR + 8u * i;
}

// Work item k of this CTA: a whole unit or, in the streamed tail, one piece
// of a unit (tiles [t0, t0 + nkv1) of its K/V sequence). Units are numbered
// head by head, so that the CTAs working at the same time share few heads
// (their K/V stay in L2). Unmasked: whole units blockIdx.x + k G (G CTAs)
// before the tail, then this CTA's tail pieces. Causal (no tail): unit 2i of
// a head is its Q block nqb-1-i and unit 2i+1 its Q block i, so that the
// pairs (2m, 2m+1) all add up to the same work; CTA c takes pairs c, c+G, ...
// slot: < 0 for a whole unit (O written out), else the part slot of a piece.
struct PItem {
  int bh, row0, t0, nkv0, nkv1, slot;
};
template <int D, bool STREAM, bool CAUSAL>
__device__ __forceinline__ bool persist_item(const FwdParams& p, int units, int k, PItem& it) {
  using C = Cfg<D>;
  const int nqb = p.N / (2 * C::BM);
  const int n = p.N / C::BN;  // K/V tiles of a whole unit (sub-tile 1 under the causal mask)
  const int G = gridDim.x, c = blockIdx.x;
  int u;
  it.t0 = 0;
  it.slot = -1;
  int t1 = n;
  if (CAUSAL) {
    const long long uu = 2ll * (c + (k / 2) * static_cast<long long>(G)) + (k & 1);
    if (uu >= units) return false;
    u = static_cast<int>(uu);
  } else {
    const int whole = STREAM ? p.st_unit0 : units;  // units handed out whole
    const long long uu = c + static_cast<long long>(k) * G;
    if (uu < whole) {
      u = static_cast<int>(uu);
    } else if (!STREAM) {
      return false;
    } else {
      if (c >= p.st_ctas) return false;
      const int rounds = c < whole ? (whole - c + G - 1) / G : 0;
      StPiece pc;
      if (!st_piece(p.st_tiles, p.st_ctas, n, c, k - rounds, pc)) return false;
      u = p.st_unit0 + pc.i;
      it.t0 = pc.t0;
      t1 = pc.t1;
      it.slot = pc.slot;
    }
  }
  it.bh = u / nqb;
  const int w = u - it.bh * nqb;
  const int qb = CAUSAL ? ((w & 1) ? w / 2 : nqb - 1 - w / 2) : w;
  it.row0 = qb * 2 * C::BM;
  if (CAUSAL) {
    // Tiles per sub-tile: up to the diagonal tile of its last row.
    it.nkv0 = (it.row0 + C::BM + C::BN - 1) / C::BN;
    it.nkv1 = (it.row0 + 2 * C::BM + C::BN - 1) / C::BN;
  } else {
    it.nkv0 = it.nkv1 = t1 - it.t0;
  }
  return true;
}

// TMA producer (one thread).
template <int D, bool STREAM, bool CAUSAL>
__device__ __forceinline__ void persist_producer(const FwdParams& p, uint32_t base, int units, const WaitCtl& ctl) {
  using C = Cfg<D>;
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);
  tma_prefetch_desc(&p.tm_o);
  const uint32_t bq = bar_addr<D>(base, C::B_Q);
  int nq = 0, g = 0;  // units whose Q was loaded; K/V tiles of the units before this one
  int gk = 0, gv = 0; // K and V loads issued (positions in the ring sequence)
  for (int kk = 0;; ++kk) {
    PItem U;
    if (!persist_item<D, STREAM, CAUSAL>(p, units, kk, U)) break;
    const int nkv = max(U.nkv0, U.nkv1);
    // The next item's Q rows into L2 while this one runs (its load, later, then hits L2).
    {
      PItem N2;
      if (persist_item<D, STREAM, CAUSAL>(p, units, kk + 1, N2)) {
        const uint16_t* qn = static_cast<const uint16_t*>(p.q) + (static_cast<size_t>(N2.bh) * p.N + N2.row0) * D;
        l2_prefetch_bulk(qn, 2u * C::Q_SUB_BYTES);
      }
    }
    // The Q buffer is free once both sub-tiles' last S products of the previous unit completed.
    if (nq > 0 && !wait_bar(xbar_addr<D>(base, PCfg<D>::X_QE), (nq - 1) & 1, ctl, kWhereQ)) break;
    mbar_arrive_expect_tx(bq, 2u * C::Q_SUB_BYTES);
    for (int sub = 0; sub < 2; ++sub)
#pragma unroll
      for (int h = 0; h < D / 64; ++h)
        tma_load_3d(base + C::OFF_Q + sub * C::Q_SUB_BYTES + h * C::Q_HALF_BYTES, &p.tm_q, bq, 64 * h,
                    U.row0 + C::BM * sub, U.bh);
    ++nq;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int gg = g + j, s = gg % C::STAGES;
      const uint32_t par = ((gg / C::STAGES) & 1) ^ 1;
      if (!wait_bar(bar_addr<D>(base, C::B_KE + s), par, ctl, kWhereKEmpty)) { ok = false; break; }
      const uint32_t kf = bar_addr<D>(base, C::B_KF + s);
      mbar_arrive_expect_tx(kf, C::KV_BYTES);
#pragma unroll
      for (int h = 0; h < D / 64; ++h)
        tma_load_3d(base + C::OFF_K + s * C::KV_BYTES + h * C::KV_HALF_BYTES, &p.tm_k, kf, 64 * h,
                    (U.t0 + j) * C::BN, U.bh);
      gk = gg + 1;
      if (!wait_bar(bar_addr<D>(base, C::B_VE + s), par, ctl, kWhereVEmpty)) { ok = false; break; }
      const uint32_t vf = bar_addr<D>(base, C::B_VF + s);
      mbar_arrive_expect_tx(vf, C::KV_BYTES);
#pragma unroll
      for (int h = 0; h < D / 64; ++h)
        tma_load_3d(base + C::OFF_V + s * C::KV_BYTES + h * C::KV_HALF_BYTES, &p.tm_v, vf, 64 * h,
                    (U.t0 + j) * C::BN, U.bh);
      gv = gg + 1;
    }
    if (!ok) break;
    g += nkv;
  }
  // Drain, always: every copy this thread started lands before the CTA exits
  // (the last Q, and the most recent tile of each ring stage).
  if (nq > 0) wait_bar_drain(bq, (nq - 1) & 1, ctl);
  for (int t = gk > C::STAGES ? gk - C::STAGES : 0; t < gk; ++t)
    wait_bar_drain(bar_addr<D>(base, C::B_KF + t % C::STAGES), (t / C::STAGES) & 1, ctl);
  for (int t = gv > C::STAGES ? gv - C::STAGES : 0; t < gv; ++t)
    wait_bar_drain(bar_addr<D>(base, C::B_VF + t % C::STAGES), (t / C::STAGES) & 1, ctl);
}

// MMA warp (whole warp; one elected lane issues): both chains' blocks of each
// unit in turn order, with positions counted across units.
template <int D, bool BF16, bool STREAM, bool CAUSAL>
__device__ __forceinline__ void persist_mma(const FwdParams& p, uint32_t base, uint32_t tmem, int units,
                                            const WaitCtl& ctl) {
  using C = Cfg<D>;
  const uint32_t b_drain = bar_addr<D>(base, C::B_DRAIN);
  int k = 0, g = 0, gp0 = 0, gp1 = 0;  // units, K/V tiles, P products of sub-tile 0 and 1 so far
  for (;; ++k) {
    PItem U;
    if (!persist_item<D, STREAM, CAUSAL>(p, units, k, U)) break;
    const int nkv = max(U.nkv0, U.nkv1);
    if (!wait_bar_warp(bar_addr<D>(base, C::B_Q), k & 1, ctl, kWhereQ)) break;
    tc_fence_after();
    bool ok = true;
    for (int j = 0; j <= nkv && ok; ++j) {
      if (j <= U.nkv0) {
        // The unit's first P.V overwrites O_0: the previous unit's epilogue must have read it.
        if (j == 1 && k > 0 && !wait_bar_warp(xbar_addr<D>(base, PCfg<D>::X_OF + 0), (k - 1) & 1, ctl, kWhereODone))
          ok = false;
        else if (!mma_block<D, BF16, 0>(p, base, tmem, j, U.nkv0, g + j, gp0 + j, ctl))
          ok = false;
      }
      if (ok && j <= U.nkv1) {
        if (j == 1 && k > 0 && !wait_bar_warp(xbar_addr<D>(base, PCfg<D>::X_OF + 1), (k - 1) & 1, ctl, kWhereODone))
          ok = false;
        else if (!mma_block<D, BF16, 1>(p, base, tmem, j, U.nkv1, g + j, gp1 + j, ctl))
          ok = false;
      }
    }
    if (!ok) break;
    g += nkv;
    gp0 += U.nkv0;
    gp1 += U.nkv1;
  }
  // All MMAs issued by this warp complete before the CTA may free TMEM / exit.
  tc_commit_elect(b_drain);
  __all_sync(0xffffffffu, wait_bar_drain(b_drain, 0, ctl));
}

// Softmax warpgroup of sub-tile `sub`: the tiles of each unit, then its
// epilogue (O / l through this sub-tile's staging buffer and TMA stores; LSE).
template <int D, bool BF16, bool STREAM, bool CAUSAL>
__device__ __forceinline__ void persist_softmax(const FwdParams& p, uint32_t base, uint32_t tmem, int sub, int units,
                                                const WaitCtl& ctl) {
  using C = Cfg<D>;
  const int t = threadIdx.x - sub * 128;  // row within the sub-tile
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = static_cast<uint32_t>(t & ~31) << 16;
  const uint32_t t_o = tmem + lane_base + (sub ? C::T_O1 : C::T_O0);
  const uint32_t t_s = tmem + lane_base + t_s_col(sub);
  const uint32_t b_od = bar_addr<D>(base, C::B_OD + sub);
  const uint32_t stage = base + PCfg<D>::OFF_STG + sub * PCfg<D>::STG_BYTES;
  const float c = p.scale * kLog2e;
  const float tau = rescale_threshold(p);
  int k = 0, g = 0, gs = 0;  // units, K/V tiles, S products of this sub-tile so far
  for (;; ++k) {
    PItem U;
    if (!persist_item<D, STREAM, CAUSAL>(p, units, k, U)) break;
    const int nkv = max(U.nkv0, U.nkv1), nkv_s = sub ? U.nkv1 : U.nkv0;
    const int my_row = U.row0 + C::BM * sub + t;
    const int row_end = CAUSAL ? min(p.N, my_row + 1) : p.N;
    float m_ref = -INFINITY, l = 0.f, l_o = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv_s; ++j) {
      // Unmasked (N a multiple of 256): every key of every tile is valid, and
      // the masked path of the tile is compiled out.
      const int valid = CAUSAL ? row_end - (U.t0 + j) * C::BN : C::BN;
      if (!softmax_tile<D, BF16>(p, base, sub, t, lane, t_s, t_o, c, tau, valid, j, g + j, gs + j, m_ref, l, l_o,
                                 ctl)) {
        ok = false;
        break;
      }
      // This sub-tile's last S product has read its Q rows.
      if (j == nkv_s - 1 && lane == 0) mbar_arrive(xbar_addr<D>(base, PCfg<D>::X_QE));
    }
    // Tiles of this unit only the other sub-tile uses: count this sub-tile's
    // stage releases once they have landed (their stage's previous phase is
    // then complete, so the arrivals cannot fall into it).
    for (int jj = nkv_s; CAUSAL && ok && jj < nkv; ++jj) {
      const int gg = g + jj, s = gg % C::STAGES;
      const uint32_t par = (gg / C::STAGES) & 1;
      ok = __all_sync(0xffffffffu, wait_bar(bar_addr<D>(base, C::B_KF + s), par, ctl, kWhereKFull) &&
                                       wait_bar(bar_addr<D>(base, C::B_VF + s), par, ctl, kWhereVFull));
      if (ok && lane == 0) {
        mbar_arrive(bar_addr<D>(base, C::B_VE + s));
        mbar_arrive(bar_addr<D>(base, C::B_KE + s));
      }
    }
    // The unit's last P.V of this sub-tile (one commit per unit); its V stage
    // is then free (d = 64: commits behind the MMAs free the stages).
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(b_od, k & 1, ctl, kWhereODone));
    if constexpr (C::SOFTMAX_FREES_STAGES)
      if (ok && lane == 0) mbar_arrive(bar_addr<D>(base, C::B_VE + (g + nkv_s - 1) % C::STAGES));
    // The whole warpgroup agrees before the epilogue, whose named barriers need all 128 threads.
    if (!named_bar_and(1 + sub, 128, ok)) break;

    tc_fence_after();
    if (STREAM && U.slot >= 0) {
      // ---- a piece of a tail unit: its normalised fp32 O and LSE to its slot ----
      const bool empty = !(l > 0.f);
      const float inv_l = empty ? 0.f : 1.0f / (BF16 ? l_o : l);
      const size_t prow = static_cast<size_t>(U.slot) * (2 * C::BM) + C::BM * sub + t;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(t_o + 32 * q, r);
        tmem_ld_wait();
        reg_fence(r);
        if (q == D / 32 - 1) {
          // O_sub has been read: the next item's first P.V may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(xbar_addr<D>(base, PCfg<D>::X_OF + sub));
        }
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D + 32 * q);
#pragma unroll
        for (int u2 = 0; u2 < 8; ++u2)
          dst[u2] = make_float4(__uint_as_float(r[4 * u2]) * inv_l, __uint_as_float(r[4 * u2 + 1]) * inv_l,
                                __uint_as_float(r[4 * u2 + 2]) * inv_l, __uint_as_float(r[4 * u2 + 3]) * inv_l);
      }
      p.lse_part[prow] = empty ? -INFINITY : (m_ref + lg2_approx(l)) * kLn2;
      g += nkv;
      gs += nkv_s;
      continue;
    }
    // ---- epilogue: O / l -> dtype -> staging (64 columns at a time) -> TMA store; LSE ----
    uint32_t pk[D / 2];
    {
      const bool empty = !(l > 0.f);
      const float inv_l = empty ? 0.f : 1.0f / (BF16 ? l_o : l);
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(t_o + 32 * q, r);
        tmem_ld_wait();
        reg_fence(r);
#pragma unroll
        for (int u2 = 0; u2 < 16; ++u2)
          pk[16 * q + u2] = pack2<BF16>(__uint_as_float(r[2 * u2]) * inv_l, __uint_as_float(r[2 * u2 + 1]) * inv_l);
      }
      // O_sub is in registers: the next unit's first P.V may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar_addr<D>(base, PCfg<D>::X_OF + sub));
      if (my_row < p.N)
        p.lse[static_cast<size_t>(U.bh) * p.N + my_row] = empty ? -INFINITY : (m_ref + lg2_approx(l)) * kLn2;
    }
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      // The previous store from this buffer must have read it.
      if (t == 0) bulk_wait_read<0>();
      named_bar_sync(1 + sub, 128);
#pragma unroll
      for (int u2 = 0; u2 < 8; ++u2) {
        const uint32_t phys = static_cast<uint32_t>(u2) ^ (static_cast<uint32_t>(t) & 7u);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + t * C::ROW_BYTES + phys * 16),
                     "r"(pk[32 * h + 4 * u2]), "r"(pk[32 * h + 4 * u2 + 1]), "r"(pk[32 * h + 4 * u2 + 2]),
                     "r"(pk[32 * h + 4 * u2 + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + sub, 128);
      if (t == 0) {
        tma_store_3d(&p.tm_o, stage, 64 * h, U.row0 + C::BM * sub, U.bh);
        tma_store_commit();
      }
    }
    g += nkv;
    gs += nkv_s;
  }
  if (t == 0) tma_store_wait_all();  // every store has completed before the CTA exits
}

template <int D, bool BF16, bool STREAM, bool CAUSAL>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1) fa_fwd_persist_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem_raw + (base - raw) + C::OFF_MISC);
  const int warp = threadIdx.x >> 5;
  // Units 0 .. units-1: all of them, or the full rounds before a split tail.
  const int units = p.qunit_count > 0 ? p.qunit_count : p.B * p.H * (p.N / (2 * C::BM));

  if (threadIdx.x == 0) {
    mbar_init(bar_addr<D>(base, C::B_Q), 1);
    // Stage releases: one arrival per softmax warp of both sub-tiles (d = 128),
    // or one commit per sub-tile's chain behind its MMAs (d = 64).
    const uint32_t rel = C::SOFTMAX_FREES_STAGES ? 8u : 2u;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_addr<D>(base, C::B_KF + s), 1);
      mbar_init(bar_addr<D>(base, C::B_KE + s), rel);
      mbar_init(bar_addr<D>(base, C::B_VF + s), 1);
      mbar_init(bar_addr<D>(base, C::B_VE + s), rel);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_addr<D>(base, C::B_SF + i), 1);
      mbar_init(bar_addr<D>(base, C::B_PF + i), 4);  // one arrival per softmax warp
      mbar_init(bar_addr<D>(base, C::B_OD + i), 1);
      mbar_init(bar_addr<D>(base, C::B_DRAIN + i), 1);
      mbar_init(xbar_addr<D>(base, PCfg<D>::X_OF + i), 4);  // one arrival per softmax warp
    }
    mbar_init(xbar_addr<D>(base, PCfg<D>::X_QE), 8);  // every softmax warp, after its last S of the unit
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
  const WaitCtl ctl{p, base + C::OFF_MISC + 4};
  // A split tail launched behind this kernel (a programmatic dependent that
  // reads none of its results) may start its CTAs as this kernel's finish.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");

  if (warp >= 8) {
    warpgroup_reg_dealloc<C::LOW_REGS>();
    if (warp == C::WARP_TMA) {
      if ((threadIdx.x & 31) == 0) persist_producer<D, STREAM, CAUSAL>(p, base, units, ctl);
      __syncwarp();
    } else if (warp == C::WARP_MMA0) {
      persist_mma<D, BF16, STREAM, CAUSAL>(p, base, tmem, units, ctl);
      __syncwarp();
    }
  } else {
    warpgroup_reg_alloc<C::HIGH_REGS>();
    persist_softmax<D, BF16, STREAM, CAUSAL>(p, base, tmem, warp / 4, units, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Whether a launch takes the persistent form: d = 128, one launch over all
// units with the whole key range (no split-KV, no key lengths), N a multiple
// of 256 (of 512 with the causal mask, whose units go in pairs) and at most
// kPersistMaxN, none of the testing build's traces. On GB300 it measured
// +2 to +5 % on B=8 H=32 N=4096 and +4 to +5 % on B=8 H=12 N=2048 against one
// CTA per unit (bit-identical results), but -6 % on B=1 H=8 N=16384: its
// tile rate is a few per cent lower (one MMA warp, runtime ring positions,
// the larger shared-memory footprint), which longer units do not win back
// from the CTA starts and ends it saves. The strict-order build keeps one
// CTA per unit.
// A streamed tail (st_ctas > 0) takes the same conditions, unmasked only,
// with its slots in o_part / lse_part and at most one range per CTA.
constexpr int kPersistMaxN = 4096;
template <int D>
bool persist_eligible(const FwdParams& p) {
#ifdef FA_STRICT_MMA_ORDER
  (void)p;
  return false;
#else
  // d = 64: unmasked launches only (its stages are freed by commits, which
  // the causal form's tiles used by one sub-tile only would not balance).
  if (D != 128 && (D != 64 || p.causal || p.st_ctas > 0)) return false;
  if (p.st_ctas > 0) {
    const long long units = static_cast<long long>(p.B) * p.H * (p.N / (2 * Cfg<D>::BM));
    if (p.causal || p.o_part == nullptr || p.lse_part == nullptr || p.st_ctas > p.num_sms || p.st_ctas > 128 ||
        p.st_unit0 < 0 ||
        p.st_unit0 >= units || p.st_unit0 % p.num_sms != 0 ||
        static_cast<long long>(p.st_tiles) != (units - p.st_unit0) * (p.N / Cfg<D>::BN) ||
        static_cast<long long>(p.st_tiles) * p.st_ctas >= (1ll << 31))
      return false;
  }
  // A launch over the first qunit_count units only (the full rounds before a
  // split tail) takes it too, unmasked: its units are then numbered in order.
  if (p.qunit_count > 0 && (p.causal || p.st_ctas > 0)) return false;
  return p.num_splits == 1 && p.qunit0 == 0 && !p.partial && p.klen == nullptr &&
         p.Nk == p.N && p.N % (p.causal ? 4 * Cfg<D>::BM : 2 * Cfg<D>::BM) == 0 && p.N <= kPersistMaxN &&
         p.stats_trace == nullptr &&
         p.timeline == nullptr &&
         p.inject == 0;
#endif
}

// Merge of the streamed tail's pieces: for each row of a tail unit cut into
// pieces, LSE = m + log sum_s exp(LSE_s - m) and O = sum_s exp(LSE_s - LSE)
// O_s over its pieces s (the block merge of the Triton page, section 2.3, in
// LSE form; m the largest LSE_s). Units that one CTA computed whole are
// skipped: their O and LSE are already written. A CTA takes 8 rows of a tail
// unit (one per warp): its first warp lists the unit's part slots in shared
// memory (one candidate range per lane), then each warp reads its row's part
// LSEs one per lane, reduces them across the warp and adds the O rows four at
// a time. Launched as a programmatic dependent of the persistent kernel: it
// lists the slots while that kernel finishes and waits for its writes before
// reading them.
constexpr int kMergeMaxPieces = 128;  // a unit has at most one piece per CTA sharing the tail (<= 126)
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_merge_stream_kernel(const __grid_constant__ FwdParams p) {
  constexpr int E = D / 32;
  static_assert(E == 4, "one float4 of O per lane and piece");
  constexpr int ROWS = 2 * Cfg<D>::BM;  // rows of a unit
  constexpr int BLOCKS_PER_UNIT = ROWS / 8;
  __shared__ int slots[kMergeMaxPieces];
  __shared__ int npieces;
  const int n = p.N / Cfg<D>::BN;
  const int i = blockIdx.x / BLOCKS_PER_UNIT;  // tail unit
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (blockIdx.x % BLOCKS_PER_UNIT) * 8 + warp;  // this warp's row of the unit
  int c_lo, c_hi;
  st_unit_ctas(p.st_tiles, p.st_ctas, n, i, c_lo, c_hi);
  if (c_lo == c_hi) return;  // whole in one range: written directly
  if (warp == 0) {
    const int x = i * n;
    int np = 0;
    for (int c0 = c_lo; c0 <= c_hi; c0 += 32) {
      const int cc = c0 + lane;
      bool has = false;
      int slot = 0;
      if (cc <= c_hi) {
        const int a = st_begin(p.st_tiles, p.st_ctas, cc);
        has = a != st_begin(p.st_tiles, p.st_ctas, cc + 1);  // an empty range holds no piece
        slot = 2 * cc + (a >= x ? 0 : 1);
      }
      const unsigned m = __ballot_sync(0xffffffffu, has);
      const int at = np + __popc(m & ((1u << lane) - 1u));
      if (has && at < kMergeMaxPieces) slots[at] = slot;
      np += __popc(m);
    }
    if (lane == 0) npieces = min(np, kMergeMaxPieces);
  }
  __syncthreads();
  const int np = npieces;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the persistent kernel's parts are written
  // the largest LSE_s, then each piece's weight w_s = exp(LSE_s - m) and their sum
  float m = -INFINITY;
  for (int s0 = lane; s0 < np; s0 += 32) m = fmaxf(m, p.lse_part[static_cast<size_t>(slots[s0]) * ROWS + r]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float acc[E] = {0.f, 0.f, 0.f, 0.f};
  float l = 0.f;
  if (m > -INFINITY) {
    for (int s0 = 0; s0 < np; s0 += 32) {
      const int cnt = min(32, np - s0);
      const float w_mine =
          lane < cnt ? ex2_approx((p.lse_part[static_cast<size_t>(slots[s0 + lane]) * ROWS + r] - m) * kLog2e) : 0.f;
      l += w_mine;
      int s = 0;
      for (; s + 4 <= cnt; s += 4) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          v[q] = reinterpret_cast<const float4*>(p.o_part + (static_cast<size_t>(slots[s0 + s + q]) * ROWS + r) * D)[lane];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float w = __shfl_sync(0xffffffffu, w_mine, s + q);
          acc[0] = fmaf(w, v[q].x, acc[0]);
          acc[1] = fmaf(w, v[q].y, acc[1]);
          acc[2] = fmaf(w, v[q].z, acc[2]);
          acc[3] = fmaf(w, v[q].w, acc[3]);
        }
      }
      for (; s < cnt; ++s) {
        const float4 v = reinterpret_cast<const float4*>(p.o_part + (static_cast<size_t>(slots[s0 + s]) * ROWS + r) * D)[lane];
        const float w = __shfl_sync(0xffffffffu, w_mine, s);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  }
  const float inv = l > 0.f ? 1.0f / l : 0.f;
  const int nqb = p.N / ROWS;
  const int u = p.st_unit0 + i;
  const long long row = static_cast<long long>(u / nqb) * p.N + (u % nqb) * ROWS + r;
  uint16_t* out = static_cast<uint16_t*>(p.o) + row * D + lane * E;
  *reinterpret_cast<uint2*>(out) = make_uint2(pack2<BF16>(acc[0] * inv, acc[1] * inv), pack2<BF16>(acc[2] * inv, acc[3] * inv));
  if (lane == 0) p.lse[row] = m > -INFINITY ? m + lg2_approx(l) * kLn2 : -INFINITY;
}

template <int D, bool BF16>
cudaError_t launch(const FwdParams& p, cudaStream_t stream) {
  using C = Cfg<D>;
  // Two instantiations: every key tile full and unmasked (its masked path
  // compiled out), or not.
  const bool full = !p.causal && p.klen == nullptr && p.Nk % C::BN == 0;
  auto kern = full ? fa_fwd_f16_kernel<D, BF16, true> : fa_fwd_f16_kernel<D, BF16, false>;
  static std::atomic<uint64_t> attr_done[2] = {0, 0};  // one bit per device ordinal (< 64)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done[full].load() & bit)) {
    // The warpgroup register split is only valid if the CTA is launched with
    // exactly LAUNCH_REGS registers per thread; otherwise refuse to launch.
    cudaFuncAttributes fa_attr;
    e = cudaFuncGetAttributes(&fa_attr, kern);
    if (e != cudaSuccess) return e;
    if (fa_attr.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[full].fetch_or(bit);
  }
  const long long all_qunits = static_cast<long long>(p.B) * p.H * ((p.N + 2 * C::BM - 1) / (2 * C::BM));
  if (p.st_ctas > 0 && !persist_eligible<D>(p)) return cudaErrorInvalidValue;
  if constexpr (D == 128 || D == 64) {
    if (persist_eligible<D>(p)) {
      // Three instantiations: unmasked, causal, unmasked with the streamed
      // tail. Each carries only its own code: the tail's item walk and part
      // epilogue cost 2-5 % of the tile rate when present (measured on GB300).
      const int variant = p.st_ctas > 0 ? 2 : p.causal ? 1 : 0;
      auto pk = fa_fwd_persist_kernel<D, BF16, false, false>;
      if constexpr (D == 128) {
        if (variant == 2) pk = fa_fwd_persist_kernel<D, BF16, true, false>;
        if (variant == 1) pk = fa_fwd_persist_kernel<D, BF16, false, true>;
      }
      static std::atomic<uint64_t> pattr[3] = {0, 0, 0};
      if (!(pattr[variant].load() & bit)) {
        cudaFuncAttributes pa;
        e = cudaFuncGetAttributes(&pa, pk);
        if (e != cudaSuccess) return e;
        if (pa.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, PCfg<D>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        pattr[variant].fetch_or(bit);
      }
      if (all_qunits <= 0 || all_qunits > 0x7fffffffLL || p.qunit_count > all_qunits) return cudaErrorInvalidValue;
      const long long units = p.qunit_count > 0 ? p.qunit_count : all_qunits;
      const long long work = p.causal ? (units + 1) / 2 : units;  // causal: pairs of units
      // With a streamed tail every SM takes part (the whole units fill rounds of num_sms).
      const long long ctas = p.st_ctas > 0 ? p.num_sms : std::min<long long>(work, p.num_sms > 0 ? p.num_sms : 1);
      pk<<<dim3(static_cast<unsigned>(ctas)), dim3(C::THREADS), PCfg<D>::SMEM_BYTES, stream>>>(p);
      e = cudaGetLastError();
      if (e != cudaSuccess || p.st_ctas == 0) return e;
      if constexpr (D == 128) {
        const long long blocks = (all_qunits - p.st_unit0) * (2 * C::BM / 8);  // 8 rows of a tail unit each
        if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
        // A programmatic dependent launch: the merge grid is set up while the
        // persistent kernel finishes and waits (griddepcontrol.wait) for its writes.
        return launch_pdl(fa_merge_stream_kernel<D, BF16>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                          p);
      }
      return cudaErrorInvalidValue;
    }
  }
  const long long qunits = p.qunit_count > 0 ? p.qunit_count : all_qunits;
  if (p.qunit0 < 0 || p.qunit0 + qunits > all_qunits) return cudaErrorInvalidValue;
  const long long units = qunits * p.num_splits;
  if (units <= 0 || units > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.launch_pdl) return launch_pdl(kern, dim3(static_cast<unsigned>(units)), dim3(C::THREADS), C::SMEM_BYTES, stream, p);
  kern<<<dim3(static_cast<unsigned>(units)), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

// Split-KV merge (block merge of the Triton page, section 2.3, in LSE form):
// LSE = m + log sum_s exp(LSE_s - m), O = sum_s exp(LSE_s - LSE) O_s, with
// m the largest LSE_s. Rows [merge_row0, B*H*N): their parts are numbered
// from merge_row0, one span per part (as the split epilogue writes them). A
// part that saw no key has LSE_s = -inf and O_s = 0 and adds nothing; a row
// that no part saw (every LSE_s = -inf: masked by the key lengths or the
// causal mask) gets O = 0 and LSE = -inf instead of 0/0 (the guard of the
// Triton page, section 5.1). One warp per output row; lane k handles D/32
// consecutive columns.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_merge_kernel(const __grid_constant__ FwdParams p) {
  constexpr int E = D / 32;
  const long long rows = static_cast<long long>(p.B) * p.H * p.N;
  const long long row = p.merge_row0 + ((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const long long span = rows - p.merge_row0, prow = row - p.merge_row0;
  float m = -INFINITY;
  for (int s = 0; s < p.num_splits; ++s) m = fmaxf(m, p.lse_part[s * span + prow]);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float l = 0.f;
  if (m > -INFINITY) {
    for (int s = 0; s < p.num_splits; ++s) {
      const float w = ex2_approx((p.lse_part[s * span + prow] - m) * kLog2e);
      l += w;
      const float* src = p.o_part + (s * span + prow) * D + lane * E;
      if constexpr (E == 8) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        const float4 y = *reinterpret_cast<const float4*>(src + 4);
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
        acc[2] = fmaf(w, x.z, acc[2]);
        acc[3] = fmaf(w, x.w, acc[3]);
        acc[4] = fmaf(w, y.x, acc[4]);
        acc[5] = fmaf(w, y.y, acc[5]);
        acc[6] = fmaf(w, y.z, acc[6]);
        acc[7] = fmaf(w, y.w, acc[7]);
      } else if constexpr (E == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
        acc[2] = fmaf(w, x.z, acc[2]);
        acc[3] = fmaf(w, x.w, acc[3]);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
      }
    }
  }
  const float inv = l > 0.f ? 1.0f / l : 0.f;
  uint32_t pk[E / 2];
#pragma unroll
  for (int e = 0; e < E / 2; ++e) pk[e] = pack2<BF16>(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  uint16_t* out = static_cast<uint16_t*>(p.o) + row * D + lane * E;
  if constexpr (E == 8)
    *reinterpret_cast<uint4*>(out) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  else if constexpr (E == 4)
    *reinterpret_cast<uint2*>(out) = make_uint2(pk[0], pk[1]);
  else
    *reinterpret_cast<uint32_t*>(out) = pk[0];
  if (lane == 0) p.lse[row] = m > -INFINITY ? m + lg2_approx(l) * kLn2 : -INFINITY;
}

template <int D, bool BF16>
cudaError_t launch_merge_t(const FwdParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.N - p.merge_row0;
  if (rows <= 0 || p.merge_row0 < 0) return cudaErrorInvalidValue;
  const long long blocks = (rows * 32 + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  fa_merge_kernel<D, BF16><<<dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const FwdParams& p, bool bf16, cudaStream_t stream) {
  if (p.d == 256) return bf16 ? launch_merge_t<256, true>(p, stream) : launch_merge_t<256, false>(p, stream);
  if (p.d == 128) return bf16 ? launch_merge_t<128, true>(p, stream) : launch_merge_t<128, false>(p, stream);
  if (p.d == 64) return bf16 ? launch_merge_t<64, true>(p, stream) : launch_merge_t<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

bool fwd_persist_eligible(const FwdParams& p) { return p.d == 128 && persist_eligible<128>(p); }

cudaError_t launch_fwd_f16(const FwdParams& p, bool bf16, cudaStream_t stream) {
  if (p.d == 128) return bf16 ? launch<128, true>(p, stream) : launch<128, false>(p, stream);
  if (p.d == 64) return bf16 ? launch<64, true>(p, stream) : launch<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
