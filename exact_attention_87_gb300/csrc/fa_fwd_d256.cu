// fa_fwd_d256.cu — FlashAttention forward for fp16 / bf16 with head dimension 256 on sm_103a.
//
// Same recurrence as the d = 64 / 128 kernel (MUSA SDK guide, "FlashAttention
// 优化", "FlashAttention 完整算法" steps 1-4: S = Q K^T per key tile, running
// row max and denominator, O rescaled by exp(m_old - m_new) before P V is
// added, O / l at the end), with the tile shape the larger head dimension
// allows (the dataflow page, section 2.1: the block size follows from the
// on-chip budget; the MUSA guide's block-size table shrinks B_c as d grows).
//
// GB300 mapping (one CTA per (batch*head, 128-row Q tile, key range), 6 warps):
//   warp 4      TMA producer: Q once (4 column blocks of 64), then K_j and V_j
//               (64 keys x 256 each) into 2-stage rings
//   warp 5      MMA warp (one elected lane issues): S_j = Q K_j^T (SS,
//               128 x 64 x 256) into one of two S buffers, O += P_j V_j (TS,
//               128 x 256 x 64: P from TMEM, V MN-major). S_{j+2} is issued
//               right behind P_j V_j, whose P it overwrites (one CTA's MMAs
//               execute in issue order), so the softmax of tile j runs while
//               S_{j+1} is on the tensor pipe
//   warps 0-3   softmax (thread = row = TMEM lane): frees K_j's stage once S_j
//               is complete, max, lazy rescale of l and O, P = 2^(s*c - m)
//               packed to 16 bits over the S columns; then
//               the epilogue (O / l through a TMA store, or under split-KV
//               this key range's fp32 O / l and LSE to the partial buffers)
// TMEM (512 columns): S0 [0,64), S1 [64,128), O [256,512). With one 128-row
// Q tile per CTA the 256 fp32 O columns fit; two Q tiles would not.
// SMEM: Q 64 KB + K ring 2 x 32 KB + V ring 2 x 32 KB.
#include <atomic>

#include "fa_device_common.cuh"
#include "fa_fwd_order.cuh"

namespace fa {
namespace {

constexpr float kLog2e256 = 1.4426950408889634f;
constexpr float kLn2_256 = 0.6931471805599453f;

struct C256 {
  static constexpr int D = 256;
  static constexpr int BM = 128;  // Q rows per CTA (TMEM lanes)
  static constexpr int BN = kD256BlockKV;  // keys per K/V tile
  static constexpr int STAGES = 2;
  static constexpr uint32_t ROW = 128;                  // one 128-byte swizzle row = 64 elements
  static constexpr uint32_t Q_BLOCK = BM * ROW;         // 64 columns of the Q tile (16 KB)
  static constexpr uint32_t Q_BYTES = 4 * Q_BLOCK;      // 64 KB
  static constexpr uint32_t KV_BLOCK = BN * ROW;        // 64 columns of a K or V tile (8 KB)
  static constexpr uint32_t KV_BYTES = 4 * KV_BLOCK;    // 32 KB
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
  static constexpr int B_Q = 0, B_KF = 1, B_KE = B_KF + STAGES, B_VF = B_KE + STAGES, B_VE = B_VF + STAGES;
  // B_OD completes once per P.V (the rescale waits for the previous one);
  // B_OL once, after the last P.V (the epilogue waits for it).
  static constexpr int B_SF = B_VE + STAGES, B_PF = B_SF + 2, B_OD = B_PF + 2, B_OL = B_OD + 1, B_DRAIN = B_OL + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_O = 256;
  static constexpr int THREADS = 192;
  static constexpr int WARP_TMA = 4, WARP_MMA = 5;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint32_t bar256(uint32_t base, int i) { return base + C256::OFF_BAR + 8u * i; }
__device__ __forceinline__ uint32_t t_s256(int buf) { return 64u * buf; }

// A descriptor the compiler must treat as computed here, so that unrolled
// k-loops do not make it hoist every k-step's descriptor into registers.
__device__ __forceinline__ uint64_t opaque256(uint64_t x) {
  asm volatile("" : "+l"(x));
  return x;
}

// --------------------------------------------------------------------------
// TMA producer (one thread)
// --------------------------------------------------------------------------
__device__ __forceinline__ void producer256(const FwdParams& p, uint32_t base, int bh, int row0, int t0, int nkv,
                                            const WaitCtl& ctl) {
  using C = C256;
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);
  tma_prefetch_desc(&p.tm_o);
  if (nkv == 0) return;  // no key to see: the epilogue writes zeros into the Q buffer
  const uint32_t bq = bar256(base, C::B_Q);
  mbar_arrive_expect_tx(bq, C::Q_BYTES);
#pragma unroll
  for (int h = 0; h < 4; ++h) tma_load_3d(base + C::OFF_Q + h * C::Q_BLOCK, &p.tm_q, bq, 64 * h, row0, bh);
  int nk = 0, nv = 0;
  bool ok = true;
  for (int j = 0; j < nkv; ++j) {
    const int s = j % C::STAGES;
    const uint32_t par = ((j / C::STAGES) & 1) ^ 1;
    if (!wait_bar(bar256(base, C::B_KE + s), par, ctl, kWhereKEmpty)) { ok = false; break; }
    const uint32_t kf = bar256(base, C::B_KF + s);
    mbar_arrive_expect_tx(kf, C::KV_BYTES);
#pragma unroll
    for (int h = 0; h < 4; ++h)
      tma_load_3d(base + C::OFF_K + s * C::KV_BYTES + h * C::KV_BLOCK, &p.tm_k, kf, 64 * h, (t0 + j) * C::BN, bh);
    nk = j + 1;
#ifdef FA_TESTING
    if (p.inject == 1 && j == 0) continue;  // fault injection: V_0 is never loaded
#endif
    if (!wait_bar(bar256(base, C::B_VE + s), par, ctl, kWhereVEmpty)) { ok = false; break; }
    const uint32_t vf = bar256(base, C::B_VF + s);
    mbar_arrive_expect_tx(vf, C::KV_BYTES);
#pragma unroll
    for (int h = 0; h < 4; ++h)
      tma_load_3d(base + C::OFF_V + s * C::KV_BYTES + h * C::KV_BLOCK, &p.tm_v, vf, 64 * h, (t0 + j) * C::BN, bh);
    nv = j + 1;
  }
  // Drain, always (the loop ended, this thread's wait gave up, or another role
  // may abort later): every copy this thread started must land before the CTA
  // exits. Cheap when nothing failed: the consumers need these copies anyway.
  (void)ok;
  {
    wait_bar_drain(bq, 0, ctl);
    for (int t = nk > C::STAGES ? nk - C::STAGES : 0; t < nk; ++t)
      wait_bar_drain(bar256(base, C::B_KF + t % C::STAGES), (t / C::STAGES) & 1, ctl);
    for (int t = nv > C::STAGES ? nv - C::STAGES : 0; t < nv; ++t) {
#ifdef FA_TESTING
      if (p.inject == 1 && t == 0) continue;  // never armed
#endif
      wait_bar_drain(bar256(base, C::B_VF + t % C::STAGES), (t / C::STAGES) & 1, ctl);
    }
  }
}

// --------------------------------------------------------------------------
// MMA warp (whole warp; one elected lane issues)
// --------------------------------------------------------------------------
template <bool BF16>
__device__ __forceinline__ void mma256(uint32_t base, uint32_t tmem, int nkv, const WaitCtl& ctl) {
  using C = C256;
  constexpr uint32_t fmt = BF16 ? 1u : 0u;
  constexpr uint32_t idesc_qk = make_idesc(fmt, 0, 0, 128, C::BN);  // S: A = Q, B = K tile, both K-major
  constexpr uint32_t idesc_pv = make_idesc(fmt, 0, 1, 128, C::D);   // O += P V: V MN-major, N = 256
  const uint32_t b_od = bar256(base, C::B_OD), b_drain = bar256(base, C::B_DRAIN);

  // S_j = Q K_j^T into S buffer j % 2 (16 k-steps over d = 256).
  auto issue_s = [&](int j) {
    const int s = j % C::STAGES;
    const uint64_t a0 = opaque256(smem_desc_sw128(base + C::OFF_Q, 16, 1024));
    const uint64_t b0 = opaque256(smem_desc_sw128(base + C::OFF_K + s * C::KV_BYTES, 16, 1024));
#pragma unroll
    for (int kk = 0; kk < C::D / 16; ++kk) {
      const uint32_t aoff = ((kk / 4) * C::Q_BLOCK + (kk & 3) * 32u) >> 4;
      const uint32_t boff = ((kk / 4) * C::KV_BLOCK + (kk & 3) * 32u) >> 4;
      mma_f16_ss_elect(tmem + t_s256(j & 1), a0 + aoff, b0 + boff, idesc_qk, kk > 0 ? 1u : 0u);
    }
    tc_commit_elect(bar256(base, C::B_SF + (j & 1)));
  };

  if (nkv == 0) goto drain;
  if (!wait_bar_warp(bar256(base, C::B_Q), 0, ctl, kWhereQ)) goto drain;
  for (int j = 0; j < nkv && j < 2; ++j) {
    if (!wait_bar_warp(bar256(base, C::B_KF + j % C::STAGES), (j / C::STAGES) & 1, ctl, kWhereKFull)) goto drain;
    tc_fence_after();
    issue_s(j);
  }
  for (int j = 0; j < nkv; ++j) {
    // O += P_j V_j (4 k-steps of 16 keys; the four 64-wide d blocks of V are 8 KB apart)
    const int s = j % C::STAGES;
    if (!wait_bar_warp(bar256(base, C::B_VF + s), (j / C::STAGES) & 1, ctl, kWhereVFull)) goto drain;
    if (!wait_bar_warp(bar256(base, C::B_PF + (j & 1)), (j / 2) & 1, ctl, kWherePFull)) goto drain;
    tc_fence_after();
    {
      const uint64_t b0 = opaque256(smem_desc_sw128(base + C::OFF_V + s * C::KV_BYTES, C::KV_BLOCK, 1024));
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_f16_ts_elect(tmem + C::T_O, tmem + t_s256(j & 1) + kk * 8, b0 + ((kk * 2048u) >> 4), idesc_pv,
                         (j > 0 || kk > 0) ? 1u : 0u);
    }
    tc_commit_elect(b_od);
    if (j == nkv - 1) tc_commit_elect(bar256(base, C::B_OL));
    tc_commit_elect(bar256(base, C::B_VE + s));
    // S_{j+2} into the columns of P_j, right behind the P_j V_j that reads them.
    if (j + 2 < nkv) {
#ifdef FA_STRICT_MMA_ORDER
      if (!wait_bar_warp(b_od, j & 1, ctl, kWhereODone)) goto drain;
#endif
      const int n = j + 2;
      if (!wait_bar_warp(bar256(base, C::B_KF + n % C::STAGES), (n / C::STAGES) & 1, ctl, kWhereKFull)) goto drain;
      tc_fence_after();
      issue_s(n);
    }
  }
drain:
  tc_commit_elect(b_drain);
  __all_sync(0xffffffffu, wait_bar_drain(b_drain, 0, ctl));
}

// --------------------------------------------------------------------------
// Softmax + lazy correction + epilogue (warps 0-3)
// --------------------------------------------------------------------------
// FULL: no key of any tile is masked (no causal mask, no key lengths, a
// multiple of 64 keys), so the masked path of the tile is compiled out.
template <bool BF16, bool FULL>
__device__ __forceinline__ void softmax256(const FwdParams& p, uint32_t base, uint32_t tmem, int bh, int row0,
                                           int split, int t0, int nkv, int key_end, const WaitCtl& ctl) {
  using C = C256;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const uint32_t lane_base = static_cast<uint32_t>(t & ~31) << 16;
  const uint32_t t_o = tmem + lane_base + C::T_O;
  const float c = p.scale * kLog2e256;
  const int my_row = row0 + t;
  const int row_end = p.causal ? min(key_end, my_row + 1) : key_end;
  const uint32_t b_od = bar256(base, C::B_OD);
  const float tau = rescale_threshold(p);
  float m_ref = -INFINITY, l = 0.f, l_o = 0.f;
  bool ok = true;

  for (int j = 0; j < nkv; ++j) {
    const uint32_t t_s = tmem + lane_base + t_s256(j & 1);
    if (!__all_sync(0xffffffffu, wait_bar(bar256(base, C::B_SF + (j & 1)), (j / 2) & 1, ctl, kWhereSFull))) {
      ok = false;
      break;
    }
    tc_fence_after();
    // S_j is complete, so K_j has been read: the softmax warps free its stage
    // (an arrival here instead of a commit behind the S MMAs, which would
    // keep the tensor pipe idle while it is processed).
    if (lane == 0) mbar_arrive(bar256(base, C::B_KE + j % C::STAGES));
    // S in registers, with each half's row max from the same load (the TMEM
    // load with a max reduction of sm_103a).
    uint32_t sraw[2][32];
    float mx_lo, mx_hi;
    tmem_ld32_max(t_s, sraw[0], mx_lo);
    tmem_ld32_max(t_s + 32, sraw[1], mx_hi);
    tmem_ld_wait();
    reg_fence(sraw[0]);
    reg_fence(sraw[1]);
    asm volatile("" : "+f"(mx_lo), "+f"(mx_hi));  // valid only after the wait, like sraw
    float s[C::BN];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      s[u] = __uint_as_float(sraw[0][u]);
      s[32 + u] = __uint_as_float(sraw[1][u]);
    }
    const int valid = FULL ? C::BN : row_end - (t0 + j) * C::BN;  // keys of this tile this row may see
    float mx = fmaxf(mx_lo, mx_hi);
    if (valid < C::BN) {
      // Masked keys become -inf and the max is taken over the rest (the
      // loads' max includes them).
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
    bool rescale_o = false;
    float alpha = 1.f;
    if (j == 0) {
      m_ref = m_new;
    } else if (__any_sync(0xffffffffu, m_new - m_ref > tau)) {
      // 0 for a row that saw no key yet (its l and O are 0), never exp2(-inf + inf)
      alpha = m_ref > -INFINITY ? ex2_approx(m_ref - m_new) : 0.f;
      m_ref = m_new;
      l *= alpha;
      l_o *= alpha;
      rescale_o = true;
    }
    // A row that has seen no key yet (every score so far masked: possible in a
    // key range of a split under the causal mask) keeps m_ref = -inf; its P
    // are taken against 0 so that they are 0, not exp2(-inf + inf).
    const float m_use = m_ref > -INFINITY ? m_ref : 0.f;
    const float2 c2 = make_float2(c, c);
    const float2 nm2 = make_float2(-m_use, -m_use);
    float2 se = make_float2(0.f, 0.f), sro = se;
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
          // Mixed-precision fp32 adds of the two rounded bf16 values (exact conversion).
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
    if (j > 0) {
      // P_{j-1} V complete, which a rescale of O needs. The wait is made at
      // every tile, not only before a rescale, so that each phase of B_OD is
      // waited for in turn and the parity always names phase j-1: P_j V
      // cannot start before this warp's P-full arrival, and the previous wait
      // saw phase j-2 complete. (S_j's completion implies that P_{j-2} V is
      // complete, but not that the commit's arrival on B_OD has landed: commits
      // on different barriers may land in any order.) P_{j-1} V normally
      // completes while this tile's softmax runs.
      if (!__all_sync(0xffffffffu, wait_bar(b_od, (j - 1) & 1, ctl, kWhereODone))) {
        ok = false;
        break;
      }
    }
    if (rescale_o) {
      tc_fence_after();
#pragma unroll 1
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
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar256(base, C::B_PF + (j & 1)));
  }
  // The last P.V, through its own barrier: a parity wait on B_OD for its
  // phase would be ambiguous while an earlier P.V is still running (only
  // the one before the previous is known complete here, from the last S).
  if (ok && nkv > 0) ok = __all_sync(0xffffffffu, wait_bar(bar256(base, C::B_OL), 0, ctl, kWhereODone));
  if (!named_bar_and(1, 128, ok)) return;

  // ---- epilogue: O / l -> dtype -> swizzled staging (Q buffer) -> TMA store; LSE ----
  tc_fence_after();
  // No key to attend to (key length 0, or under the causal mask no key of
  // this split's range for this row): O = 0, LSE = -inf instead of 0/0.
  const bool empty = nkv == 0 || !(l > 0.f);
  const float inv_l = empty ? 0.f : 1.0f / (BF16 ? l_o : l);
  if (p.num_splits > 1 || p.partial) {
    // Split-KV (or one part of a merge done elsewhere): this key range's
    // normalised O (fp32) and LSE go to the partial buffers, rows numbered
    // from merge_row0, one span of rows per key range.
    const size_t span = static_cast<size_t>(p.B) * p.H * p.N - p.merge_row0;
    const size_t prow = static_cast<size_t>(split) * span + (static_cast<size_t>(bh) * p.N + my_row - p.merge_row0);
#pragma unroll 1
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
    if (my_row < p.N) p.lse_part[prow] = empty ? -INFINITY : (m_ref + lg2_approx(l)) * kLn2_256;
    return;
  }
  const uint32_t stage = base + C::OFF_Q;
#pragma unroll 1
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
    const uint32_t blk = q / 2, chunk0 = (q & 1) * 4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t phys = (chunk0 + u) ^ (static_cast<uint32_t>(t) & 7u);
      const uint32_t addr = stage + blk * C::Q_BLOCK + t * C::ROW + phys * 16;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * u]), "r"(pk[4 * u + 1]),
                   "r"(pk[4 * u + 2]), "r"(pk[4 * u + 3])
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  named_bar_sync(1, 128);
  if (t == 0) {
#pragma unroll
    for (int h = 0; h < 4; ++h) tma_store_3d(&p.tm_o, stage + h * C::Q_BLOCK, 64 * h, row0, bh);
    tma_store_commit();
    tma_store_wait_all();
  }
  if (my_row < p.N)
    p.lse[static_cast<size_t>(bh) * p.N + my_row] = empty ? -INFINITY : (m_ref + lg2_approx(l)) * kLn2_256;
}

template <bool BF16, bool FULL>
__global__ void __launch_bounds__(C256::THREADS, 1) fa_fwd_d256_kernel(const __grid_constant__ FwdParams p) {
  using C = C256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem_raw + (base - raw) + C::OFF_MISC);
  const int warp = threadIdx.x >> 5;
  // Work unit: (batch*head, 128-row Q tile, key range), in the order of
  // fa_fwd_order.cuh: a head's Q tiles in a row; causal launches over every
  // unit unsplit, longest first within windows of heads. Split launches keep
  // the natural order, in which the units of the split-KV tail plan (the
  // last ones) hold the last rows: its merge and partial buffers cover the
  // rows from merge_row0 on.
  const int nqb = (p.N + C::BM - 1) / C::BM;
  const int split = blockIdx.x % p.num_splits;
  const int qunit = p.qunit0 + blockIdx.x / p.num_splits;
  const bool heavy_first = p.causal && p.num_splits == 1 && p.qunit_count == 0;
  const FwdUnitOf unit = fwd_unit_of(qunit, p.B * p.H, nqb, p.Nk, 256, heavy_first, p.num_sms);
  const int bh = unit.bh;
  const int qb = unit.qb;
  const int row0 = qb * C::BM;
  // Keys this unit may see: [0, key_end); causal limits the tile to its own last row.
  const int key_end = p.klen ? max(0, min(p.Nk, p.klen[bh / p.H])) : p.Nk;
  const int end = p.causal ? min(key_end, row0 + C::BM) : key_end;
  const int t0 = split * p.split_tiles;  // first K/V tile of this key range
  // Tiles in this key range (none when the unit's keys end before the range starts).
  const int nkv = max(0, min((end + C::BN - 1) / C::BN - t0, p.split_tiles));

  if (threadIdx.x == 0) {
    mbar_init(bar256(base, C::B_Q), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar256(base, C::B_KF + s), 1);
      mbar_init(bar256(base, C::B_KE + s), 4);  // one arrival per softmax warp
      mbar_init(bar256(base, C::B_VF + s), 1);
      mbar_init(bar256(base, C::B_VE + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar256(base, C::B_SF + i), 1);
      mbar_init(bar256(base, C::B_PF + i), 4);  // one arrival per softmax warp
    }
    mbar_init(bar256(base, C::B_OD), 1);
    mbar_init(bar256(base, C::B_OL), 1);
    mbar_init(bar256(base, C::B_DRAIN), 1);
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
  const WaitCtl ctl{p, base + C::OFF_MISC + 4};
  // A split tail launched behind this kernel (a programmatic dependent that
  // reads none of its results) may start its CTAs as this kernel's finish.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");

  if (warp == C::WARP_TMA) {
    if ((threadIdx.x & 31) == 0) producer256(p, base, bh, row0, t0, nkv, ctl);
    __syncwarp();
  } else if (warp == C::WARP_MMA) {
    mma256<BF16>(base, tmem, nkv, ctl);
    __syncwarp();
  } else {
    softmax256<BF16, FULL>(p, base, tmem, bh, row0, split, t0, nkv, key_end, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // Launched as a programmatic dependent (the split tail after the full
  // waves): finish only after the kernel before it (no-op otherwise).
  if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <bool BF16>
cudaError_t launch256(const FwdParams& p, cudaStream_t stream) {
  using C = C256;
  // Two instantiations: every key tile full and unmasked (its masked path
  // compiled out), or not.
  const bool full = !p.causal && p.klen == nullptr && p.Nk % C::BN == 0;
  auto kern = full ? fa_fwd_d256_kernel<BF16, true> : fa_fwd_d256_kernel<BF16, false>;
  static std::atomic<uint64_t> attr_done[2] = {0, 0};  // one bit per device ordinal (< 64)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done[full].load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[full].fetch_or(bit);
  }
  const long long all_qunits = static_cast<long long>(p.B) * p.H * ((p.N + C::BM - 1) / C::BM);
  const long long qunits = p.qunit_count > 0 ? p.qunit_count : all_qunits;
  if (p.qunit0 < 0 || p.qunit0 + qunits > all_qunits) return cudaErrorInvalidValue;
  const long long units = qunits * p.num_splits;
  if (units <= 0 || units > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.launch_pdl) return launch_pdl(kern, dim3(static_cast<unsigned>(units)), dim3(C::THREADS), C::SMEM_BYTES, stream, p);
  kern<<<dim3(static_cast<unsigned>(units)), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d256(const FwdParams& p, bool bf16, cudaStream_t stream) {
  return bf16 ? launch256<true>(p, stream) : launch256<false>(p, stream);
}

}  // namespace fa
