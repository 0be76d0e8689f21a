// fa_bwd_d256.cu — FlashAttention backward pass (dQ, dK, dV) for fp16 / bf16
// with head dimension 256 on sm_103a.
//
// The same recomputation as the d = 64 / 128 backward (the MUSA SDK guide,
// "重计算（Recompute）换存储"; the Triton page, sections 2.4 and 4.4):
//     P_ij  = exp(s_ij - LSE_i),        s_ij = scale * q_i . k_j
//     dV_j  = sum_i P_ij dO_i
//     dS_ij = P_ij (dO_i . v_j - D_i)
//     dQ_i  = scale * sum_j dS_ij k_j,  dK_j = scale * sum_i dS_ij q_i
// with the row statistics (D_i, LSE_i * log2 e) and the fp32 dQ accumulator
// prepared, and dQ rounded at the end, by the kernels of fa_bwd_f16.cu.
//
// Why two passes. A CTA owns a 128-key tile and accumulates dK_j and dV_j
// over every Q tile; at d = 256 each accumulator is 128 x 256 fp32, i.e. 256
// of the 512 TMEM columns, so dK and dV together fill TMEM and leave nothing
// for S^T and dP^T (the dataflow page, section 2.1: the tile shape follows the
// on-chip budget). The work is therefore split over two kernels, each with
// one accumulator:
//   fa_bwd_dv256   dV_j = sum_i P^T_ij dO_i    (S^T recomputed; no dP, no dS)
//   fa_bwd_dkdq256 dK_j and the dQ_i contributions (S^T, dP^T, dS)
// so S^T is computed twice: 6 products per (key tile, Q tile) instead of 5.
// Shared memory sets the Q tile at 64 rows (a 64 x 256 16-bit Q or dO tile is
// 32 KB; K and V stay resident at 64 KB each).
//
// fa_bwd_dv256 (6 warps; TMEM lanes = keys):
//   warp 4      TMA producer: K_j once; Q_i (+ its LSE * log2 e row) and dO_i
//               into 2-stage rings
//   warp 5      MMA warp: S^T_i = K_j Q_i^T (SS, 128 x 64 x 256) into one of
//               two S buffers; dV += P^T_i dO_i (TS, 128 x 256 x 64: P^T from
//               TMEM, dO MN-major). S^T_{i+2} is issued right behind dV_i,
//               whose P^T it overwrites (one CTA's MMAs execute in issue
//               order; -DFA_STRICT_MMA_ORDER waits for dV_i instead), so the
//               softmax of tile i runs while S^T_{i+1} is on the tensor pipe
//   warps 0-3   thread = key: P = 2^(s * scale * log2 e - LSE_i * log2 e),
//               packed to 16 bits over the first 32 columns of its S buffer;
//               they free each Q stage once they have read its LSE row; at
//               the end dV_j -> 16-bit -> TMA store
//   TMEM: S^T buffers [0,64) and [64,128), dV [256,512).
//
// fa_bwd_dkdq256 (12 warps; TMEM lanes = keys, and d for dQ^T):
//   warp 8      TMA producer: K_j, V_j once; Q_i (+ LSE and D rows) and dO_i,
//               one stage each
//   warp 9      MMA warp, per Q tile i:
//                 dP^T_i = V_j dO_i^T   (SS, 128 x 64 x 256)
//                 S^T_i  = K_j Q_i^T    (SS, 128 x 64 x 256)
//                 dK    += dS^T_i Q_i   (SS, 128 x 256 x 64: Q MN-major)
//                 dQ^T_i = K_j^T dS^T_i (SS, two 128 x 64 x 128 halves of d:
//                                        K and dS^T both read MN-major)
//               dP^T_{i+1} is issued as soon as the softmax has read dP^T_i,
//               so it runs while dS_i is formed
//   warps 0-3   thread = key: P from S^T_i, dS^T * scale = P * scale *
//               (dP^T - D) rounded to 16 bits into the dS^T tile in SMEM; at
//               the end dK_j -> 16-bit -> TMA store
//   warps 4-7   dQ: thread = column d of a half; both halves of dQ^T_i from
//               TMEM into registers (which frees the columns), then one fp32
//               reduction per element into the dQ accumulator (the 32 lanes
//               of a warp cover 32 consecutive columns of one row)
//   warps 10-11 idle (complete the third warpgroup)
//   TMEM: S^T [0,64), dP^T [64,128), dQ^T [128,256), dK [256,512).
#include <atomic>
#include <type_traits>

#include "fa_bwd_order.cuh"
#include "fa_device_common.cuh"

namespace fa {
namespace {

constexpr float kLog2eD = 1.4426950408889634f;
using DCtl = WaitCtlT<BwdParams>;

// Shapes common to both passes.
struct B256 {
  static constexpr int D = 256;
  static constexpr int BK = 128;                // keys per CTA (TMEM lanes, MMA M)
  static constexpr int BQ = 64;                 // queries per Q tile (MMA N of S^T, dP^T)
  static constexpr uint32_t ROW = 128;          // one 128-byte swizzle row = 64 16-bit elements
  static constexpr uint32_t KBLK = BK * ROW;    // 64 columns of a K or V tile (16 KB)
  static constexpr uint32_t KTILE = 4 * KBLK;   // a K or V tile (64 KB)
  static constexpr uint32_t QBLK = BQ * ROW;    // 64 columns of a Q or dO tile (8 KB)
  static constexpr uint32_t QTILE = 4 * QBLK;   // a Q or dO tile (32 KB)
  static constexpr uint32_t ROWS = BQ * 4;      // one fp32 row statistic of a Q tile (256 bytes)
};

// fa_bwd_dv256 shared memory and barriers.
struct CA : B256 {
  static constexpr int ST = 2;  // Q and dO stages
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_Q = OFF_K + KTILE;
  static constexpr uint32_t OFF_DO = OFF_Q + ST * QTILE;
  static constexpr uint32_t OFF_ROWS = OFF_DO + ST * QTILE;  // [ST] x lse2[64]
  static constexpr uint32_t OFF_BAR = OFF_ROWS + ST * ROWS;
  static constexpr int B_K = 0, B_QF = 1, B_QE = B_QF + ST, B_OF = B_QE + ST, B_OE = B_OF + ST;
  static constexpr int B_SF = B_OE + ST, B_PF = B_SF + 2, B_DONE = B_PF + 2, B_DRAIN = B_DONE + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_DV = 256;
  static constexpr int THREADS = 192;
  static constexpr int WARP_TMA = 4, WARP_MMA = 5;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// fa_bwd_dkdq256 shared memory and barriers.
struct CB : B256 {
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KTILE;
  static constexpr uint32_t OFF_Q = OFF_V + KTILE;
  static constexpr uint32_t OFF_DO = OFF_Q + QTILE;
  static constexpr uint32_t OFF_DS = OFF_DO + QTILE;        // dS^T: 128 keys x 64 queries, 16-bit (16 KB)
  static constexpr uint32_t OFF_ROWS = OFF_DS + BK * ROW;   // lse2[64], dsum[64]
  static constexpr uint32_t OFF_BAR = OFF_ROWS + 2 * ROWS;
  static constexpr int B_K = 0, B_V = 1, B_QF = 2, B_QE = 3, B_OF = 4, B_OE = 5, B_SF = 6, B_DPF = 7;
  static constexpr int B_SC = 8, B_DSF = 9, B_DSE = 10, B_DQF = 11, B_DQE = 12, B_DONE = 13, B_DRAIN = 14;
  static constexpr int NBAR = 15;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DP = 64, T_DQ = 128, T_DK = 256;
  static constexpr int THREADS = 384;
  static constexpr int WARP_TMA = 8, WARP_MMA = 9;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <class C>
__device__ __forceinline__ uint32_t dbar(uint32_t base, int i) {
  return base + C::OFF_BAR + 8u * i;
}

// A descriptor the compiler must treat as computed here, so that unrolled
// k-loops do not make it hoist every k-step's descriptor into registers.
__device__ __forceinline__ uint64_t opaque_d(uint64_t x) {
  asm volatile("" : "+l"(x));
  return x;
}

// M x N x 256 product of two K-major tiles in 128-byte swizzle: A has its four
// 64-column blocks a_blk bytes apart, B b_blk bytes apart (16 k-steps of 16).
__device__ __forceinline__ void mma_kmajor_d256(uint32_t d_tmem, uint32_t a_base, uint32_t a_blk, uint32_t b_base,
                                                uint32_t b_blk, uint32_t idesc) {
  const uint64_t a0 = opaque_d(smem_desc_sw128(a_base, 16, 1024));
  const uint64_t b0 = opaque_d(smem_desc_sw128(b_base, 16, 1024));
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const uint32_t aoff = ((kk / 4) * a_blk + (kk & 3) * 32u) >> 4;
    const uint32_t boff = ((kk / 4) * b_blk + (kk & 3) * 32u) >> 4;
    mma_f16_ss_elect(d_tmem, a0 + aoff, b0 + boff, idesc, kk > 0 ? 1u : 0u);
  }
}

// Keys this CTA sees and the Q tiles it visits (both passes): with the causal
// mask the Q tiles before the key tile's first row see none of its keys.
struct KeyTile {
  int bh, kv0, key_end, q_first, nq;
};
__device__ __forceinline__ KeyTile key_tile(const BwdParams& p) {
  KeyTile k;
  const int nt = (p.N + B256::BK - 1) / B256::BK;
  const BwdTileOf tile = bwd_tile_of(static_cast<int>(blockIdx.x), p.B * p.H, nt, p.N, B256::D, p.causal != 0);
  k.bh = tile.bh;
  k.kv0 = tile.kt * B256::BK;
  k.key_end = p.klen != nullptr ? min(max(p.klen[k.bh / p.H], 0), p.N) : p.N;
  k.q_first = p.causal ? k.kv0 / B256::BQ : 0;
  k.nq = k.kv0 < k.key_end ? (p.N + B256::BQ - 1) / B256::BQ - k.q_first : 0;
  return k;
}

// Zero dK or dV rows [kv0, kv0 + 128) of a key tile that no query sees.
__device__ __forceinline__ void zero_key_rows(const BwdParams& p, void* dst, const KeyTile& kt, int nthreads) {
  const int rows = min(B256::BK, p.N - kt.kv0);
  const long long first = (static_cast<long long>(kt.bh) * p.N + kt.kv0) * B256::D;  // 16-bit elements
  uint4* z = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + first);
  for (int x = threadIdx.x; x < rows * B256::D / 8; x += nthreads) z[x] = make_uint4(0u, 0u, 0u, 0u);
}

// Per thread (key t of the tile): P of query column c of Q tile qt is forced
// to 0 when c < limit (the causal mask: query 64*qt + c sees key kv0 + t only
// if kv0 + t <= 64*qt + c; a key past the key length: every column).
__device__ __forceinline__ int mask_limit(const BwdParams& p, const KeyTile& kt, int t, int qt) {
  if (kt.kv0 + t >= kt.key_end) return B256::BQ;
  return p.causal ? max(0, min(B256::BQ, kt.kv0 + t - B256::BQ * qt)) : 0;
}
// Whether Q tile qt has any masked entry in this CTA (uniform over the CTA).
__device__ __forceinline__ bool tile_masked(const BwdParams& p, const KeyTile& kt, int qt) {
  return kt.kv0 + B256::BK > kt.key_end || (p.causal && kt.kv0 + B256::BK - 1 > B256::BQ * qt);
}

// P for one thread's key over the 64 queries of a Q tile, from its S^T row
// (rs), the tile's LSE * log2 e row (lse2) and the mask limit; 16-bit pairs
// into pk (queries 2u, 2u+1 -> pk[u]) and, with SCALED, P * scale into ps.
template <bool BF16, bool MASKED, bool SCALED>
__device__ __forceinline__ void p_row(const uint32_t (&rs)[2][32], const float* lse2, float c, float scale, int lim,
                                      uint32_t (&pk)[32], float* ps) {
  const float2 c2 = make_float2(c, c);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 l4 = reinterpret_cast<const float4*>(lse2)[8 * q + u];
      const uint32_t (&r)[32] = rs[q];
      const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1])), c2,
                                   make_float2(-l4.x, -l4.y));
      const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])), c2,
                                   make_float2(-l4.z, -l4.w));
      float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
      float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
      if constexpr (MASKED) {
        const int c0 = 32 * q + 4 * u;
        if (c0 < lim) p0.x = 0.f;
        if (c0 + 1 < lim) p0.y = 0.f;
        if (c0 + 2 < lim) p1.x = 0.f;
        if (c0 + 3 < lim) p1.y = 0.f;
      }
      pk[16 * q + 2 * u] = pack2<BF16>(p0.x, p0.y);
      pk[16 * q + 2 * u + 1] = pack2<BF16>(p1.x, p1.y);
      if constexpr (SCALED) {
        ps[32 * q + 4 * u] = p0.x * scale;
        ps[32 * q + 4 * u + 1] = p0.y * scale;
        ps[32 * q + 4 * u + 2] = p1.x * scale;
        ps[32 * q + 4 * u + 3] = p1.y * scale;
      }
    }
  }
}

// A 128 x 256 fp32 TMEM accumulator (this thread's lane = row t) as a 16-bit
// tile: swizzled staging at `stage` (four 16 KB blocks of 64 columns), then TMA.
template <bool BF16>
__device__ __forceinline__ void store_acc256(uint32_t t_acc, uint32_t stage, int t, int bar_id, const CUtensorMap* map,
                                             int row0, int bh) {
#pragma unroll 1
  for (int q = 0; q < 8; ++q) {
    uint32_t r[32];
    tmem_ld32(t_acc + 32 * q, r);
    tmem_ld_wait();
    reg_fence(r);
    uint32_t pk[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) pk[u] = pack2<BF16>(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
    const uint32_t blk = q / 2, chunk0 = (q & 1) * 4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t phys = (chunk0 + u) ^ (static_cast<uint32_t>(t) & 7u);
      const uint32_t addr = stage + blk * B256::KBLK + t * B256::ROW + phys * 16;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * u]), "r"(pk[4 * u + 1]),
                   "r"(pk[4 * u + 2]), "r"(pk[4 * u + 3])
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  named_bar_sync(bar_id, 128);
  if (t == 0) {
#pragma unroll
    for (int h = 0; h < 4; ++h) tma_store_3d(map, stage + h * B256::KBLK, 64 * h, row0, bh);
    tma_store_commit();
    tma_store_wait_all();
  }
}

// ==========================================================================
// fa_bwd_dv256
// ==========================================================================
// TMA producer (one thread): K once, then Q_i with its LSE row and dO_i.
__device__ __forceinline__ void dv_producer(const BwdParams& p, uint32_t base, const KeyTile& kt, const DCtl& ctl) {
  using C = CA;
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_do);
  const uint32_t bk = dbar<C>(base, C::B_K);
  mbar_arrive_expect_tx(bk, C::KTILE);
#pragma unroll
  for (int h = 0; h < 4; ++h) tma_load_3d(base + C::OFF_K + h * C::KBLK, &p.tm_k, bk, 64 * h, kt.kv0, kt.bh);
  const size_t row_base = static_cast<size_t>(kt.bh) * p.n_pad;
  int nqi = 0, noi = 0;  // Q / dO tiles whose loads were issued
  for (int i = 0; i < kt.nq; ++i) {
    const int s = i % C::ST;
    const uint32_t par = ((i / C::ST) & 1) ^ 1;
    const int q0 = (kt.q_first + i) * C::BQ;
    if (!wait_bar(dbar<C>(base, C::B_QE + s), par, ctl, kWhereBwdQEmpty)) break;
    const uint32_t qf = dbar<C>(base, C::B_QF + s);
    mbar_arrive_expect_tx(qf, C::QTILE + C::ROWS);
#pragma unroll
    for (int h = 0; h < 4; ++h) tma_load_3d(base + C::OFF_Q + s * C::QTILE + h * C::QBLK, &p.tm_q, qf, 64 * h, q0, kt.bh);
    bulk_load(base + C::OFF_ROWS + s * C::ROWS, p.lse2 + row_base + q0, C::ROWS, qf);
    nqi = i + 1;
    if (!wait_bar(dbar<C>(base, C::B_OE + s), par, ctl, kWhereBwdDoEmpty)) break;
    const uint32_t of = dbar<C>(base, C::B_OF + s);
    mbar_arrive_expect_tx(of, C::QTILE);
#pragma unroll
    for (int h = 0; h < 4; ++h)
      tma_load_3d(base + C::OFF_DO + s * C::QTILE + h * C::QBLK, &p.tm_do, of, 64 * h, q0, kt.bh);
    noi = i + 1;
  }
  // Drain, always: every copy this thread started lands before the CTA exits.
  wait_bar_drain(bk, 0, ctl);
  for (int t = nqi > C::ST ? nqi - C::ST : 0; t < nqi; ++t)
    wait_bar_drain(dbar<C>(base, C::B_QF + t % C::ST), (t / C::ST) & 1, ctl);
  for (int t = noi > C::ST ? noi - C::ST : 0; t < noi; ++t)
    wait_bar_drain(dbar<C>(base, C::B_OF + t % C::ST), (t / C::ST) & 1, ctl);
}

// MMA warp: S^T_i into buffer i % 2, dV += P^T_i dO_i, S^T_{i+2} right behind dV_i.
template <bool BF16>
__device__ __forceinline__ void dv_mma(uint32_t base, uint32_t tmem, int nq, const DCtl& ctl) {
  using C = CA;
  constexpr uint32_t fmt = BF16 ? 1u : 0u;
  constexpr uint32_t idesc_s = make_idesc(fmt, 0, 0, 128, C::BQ);  // S^T: A = K (M = keys), B = Q, both K-major
  constexpr uint32_t idesc_dv = make_idesc(fmt, 0, 1, 128, C::D);  // dV: B = dO with d contiguous (MN-major)
  const uint32_t b_drain = dbar<C>(base, C::B_DRAIN);
  auto issue_s = [&](int i) {
    mma_kmajor_d256(tmem + 64u * (i & 1), base + C::OFF_K, C::KBLK, base + C::OFF_Q + (i % C::ST) * C::QTILE,
                    C::QBLK, idesc_s);
    tc_commit_elect(dbar<C>(base, C::B_SF + (i & 1)));
  };
  if (nq == 0) goto drain;
  if (!wait_bar_warp(dbar<C>(base, C::B_K), 0, ctl, kWhereBwdKV)) goto drain;
  for (int i = 0; i < nq && i < 2; ++i) {
    if (!wait_bar_warp(dbar<C>(base, C::B_QF + i % C::ST), (i / C::ST) & 1, ctl, kWhereBwdQFull)) goto drain;
    tc_fence_after();
    issue_s(i);
  }
  for (int i = 0; i < nq; ++i) {
    const int s = i % C::ST;
    if (!wait_bar_warp(dbar<C>(base, C::B_OF + s), (i / C::ST) & 1, ctl, kWhereBwdDoFull)) goto drain;
    if (!wait_bar_warp(dbar<C>(base, C::B_PF + (i & 1)), (i / 2) & 1, ctl, kWhereBwdPFull)) goto drain;
    tc_fence_after();
    {
      // 4 k-steps of 16 queries: P^T packed in columns [8kk, 8kk+8) of the
      // buffer; dO's 16 rows are two 8-row swizzle atoms (2048 bytes), its
      // four 64-wide d blocks 8 KB apart.
      const uint64_t b0 = opaque_d(smem_desc_sw128(base + C::OFF_DO + s * C::QTILE, C::QBLK, 1024));
#pragma unroll
      for (int kk = 0; kk < C::BQ / 16; ++kk)
        mma_f16_ts_elect(tmem + C::T_DV, tmem + 64u * (i & 1) + 8 * kk, b0 + ((kk * 2048u) >> 4), idesc_dv,
                         (i > 0 || kk > 0) ? 1u : 0u);
    }
    tc_commit_elect(dbar<C>(base, C::B_OE + s));
    if (i == nq - 1) tc_commit_elect(dbar<C>(base, C::B_DONE));
    if (i + 2 < nq) {
      const int n = i + 2;
#ifdef FA_STRICT_MMA_ORDER
      // S^T_{i+2} overwrites P^T_i: the strict build waits for dV_i to complete.
      if (!wait_bar_warp(dbar<C>(base, C::B_OE + s), (i / C::ST) & 1, ctl, kWhereBwdDoEmpty)) goto drain;
#endif
      if (!wait_bar_warp(dbar<C>(base, C::B_QF + n % C::ST), (n / C::ST) & 1, ctl, kWhereBwdQFull)) goto drain;
      tc_fence_after();
      issue_s(n);
    }
  }
drain:
  tc_commit_elect(b_drain);
  __all_sync(0xffffffffu, wait_bar_drain(b_drain, 0, ctl));
}

// Softmax warps 0-3 (thread = key): P^T_i over its S buffer; at the end dV.
template <bool BF16>
__device__ __forceinline__ void dv_softmax(const BwdParams& p, const uint8_t* smem, uint32_t base, uint32_t tmem,
                                           const KeyTile& kt, const DCtl& ctl) {
  using C = CA;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const uint32_t lane_base = static_cast<uint32_t>(t & ~31) << 16;
  const float c = p.scale * kLog2eD;
  bool ok = true;
  for (int i = 0; i < kt.nq; ++i) {
    const int s = i % C::ST, b = i & 1, qt = kt.q_first + i;
    const uint32_t t_s = tmem + lane_base + 64u * b;
    if (!named_bar_and(1, 128, wait_bar(dbar<C>(base, C::B_SF + b), (i / 2) & 1, ctl, kWhereBwdSFull))) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t rs[2][32];
    tmem_ld32(t_s, rs[0]);
    tmem_ld32(t_s + 32, rs[1]);
    tmem_ld_wait();
    reg_fence(rs[0]);
    reg_fence(rs[1]);
    const float* lse2 = reinterpret_cast<const float*>(smem + C::OFF_ROWS + s * C::ROWS);
    uint32_t pk[32];
    if (tile_masked(p, kt, qt))
      p_row<BF16, true, false>(rs, lse2, c, 0.f, mask_limit(p, kt, t, qt), pk, nullptr);
    else
      p_row<BF16, false, false>(rs, lse2, c, 0.f, 0, pk, nullptr);
    // Queries 2u, 2u+1 -> packed column u of the buffer (the A operand of dV).
    uint32_t lo[16], hi[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      lo[u] = pk[u];
      hi[u] = pk[16 + u];
    }
    tmem_st16(t_s, lo);
    tmem_st16(t_s + 16, hi);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(dbar<C>(base, C::B_PF + b));
      // S^T_i has read Q_i, and this warp has read the LSE row: the stage is free.
      mbar_arrive(dbar<C>(base, C::B_QE + s));
    }
  }
  if (ok && kt.nq > 0) ok = wait_bar(dbar<C>(base, C::B_DONE), 0, ctl, kWhereBwdDone);
  if (!named_bar_and(1, 128, ok)) return;
  tc_fence_after();
  // Every MMA is complete: the K tile's shared memory stages dV.
  store_acc256<BF16>(tmem + lane_base + C::T_DV, base + C::OFF_K, t, 1, &p.tm_dv, kt.kv0, kt.bh);
}

template <bool BF16>
__global__ void __launch_bounds__(CA::THREADS, 1) fa_bwd_dv256_kernel(const __grid_constant__ BwdParams p) {
  using C = CA;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5;
  const KeyTile kt = key_tile(p);
  if (kt.nq == 0) {
    // Every key of this tile is masked: its dV rows are zero. Nothing has been set up yet.
    zero_key_rows(p, p.dv, kt, C::THREADS);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(dbar<C>(base, C::B_K), 1);
    for (int s = 0; s < C::ST; ++s) {
      mbar_init(dbar<C>(base, C::B_QF + s), 1);
      mbar_init(dbar<C>(base, C::B_QE + s), 4);  // one arrival per softmax warp
      mbar_init(dbar<C>(base, C::B_OF + s), 1);
      mbar_init(dbar<C>(base, C::B_OE + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(dbar<C>(base, C::B_SF + b), 1);
      mbar_init(dbar<C>(base, C::B_PF + b), 4);  // one arrival per softmax warp
    }
    mbar_init(dbar<C>(base, C::B_DONE), 1);
    mbar_init(dbar<C>(base, C::B_DRAIN), 1);
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
  const DCtl ctl{p, base + C::OFF_MISC + 4};
  if (warp == C::WARP_TMA) {
    if ((threadIdx.x & 31) == 0) dv_producer(p, base, kt, ctl);
    __syncwarp();
  } else if (warp == C::WARP_MMA) {
    dv_mma<BF16>(base, tmem, kt.nq, ctl);
    __syncwarp();
  } else {
    dv_softmax<BF16>(p, smem, base, tmem, kt, ctl);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ==========================================================================
// fa_bwd_dkdq256
// ==========================================================================
// TMA producer (one thread): K, V once, then dO_i and Q_i (+ LSE and D rows),
// one stage each (dO_i is freed by dP^T_i, Q_i only by dK_i).
__device__ __forceinline__ void dkdq_producer(const BwdParams& p, uint32_t base, const KeyTile& kt, const DCtl& ctl) {
  using C = CB;
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);
  tma_prefetch_desc(&p.tm_do);
  const uint32_t bk = dbar<C>(base, C::B_K), bv = dbar<C>(base, C::B_V);
  mbar_arrive_expect_tx(bk, C::KTILE);
#pragma unroll
  for (int h = 0; h < 4; ++h) tma_load_3d(base + C::OFF_K + h * C::KBLK, &p.tm_k, bk, 64 * h, kt.kv0, kt.bh);
  mbar_arrive_expect_tx(bv, C::KTILE);
#pragma unroll
  for (int h = 0; h < 4; ++h) tma_load_3d(base + C::OFF_V + h * C::KBLK, &p.tm_v, bv, 64 * h, kt.kv0, kt.bh);
  const size_t row_base = static_cast<size_t>(kt.bh) * p.n_pad;
  const uint32_t qf = dbar<C>(base, C::B_QF), of = dbar<C>(base, C::B_OF);
  int nqi = 0, noi = 0;
  for (int i = 0; i < kt.nq; ++i) {
    const uint32_t par = (i & 1) ^ 1;
    const int q0 = (kt.q_first + i) * C::BQ;
#ifdef FA_TESTING
    if (!(p.inject == 1 && i == 0)) {  // fault injection: dO_0 is never loaded
#endif
      if (!wait_bar(dbar<C>(base, C::B_OE), par, ctl, kWhereBwdDoEmpty)) break;
      mbar_arrive_expect_tx(of, C::QTILE);
#pragma unroll
      for (int h = 0; h < 4; ++h) tma_load_3d(base + C::OFF_DO + h * C::QBLK, &p.tm_do, of, 64 * h, q0, kt.bh);
      noi = i + 1;
#ifdef FA_TESTING
    }
#endif
    if (!wait_bar(dbar<C>(base, C::B_QE), par, ctl, kWhereBwdQEmpty)) break;
    mbar_arrive_expect_tx(qf, C::QTILE + 2 * C::ROWS);
#pragma unroll
    for (int h = 0; h < 4; ++h) tma_load_3d(base + C::OFF_Q + h * C::QBLK, &p.tm_q, qf, 64 * h, q0, kt.bh);
    bulk_load(base + C::OFF_ROWS, p.lse2 + row_base + q0, C::ROWS, qf);
    bulk_load(base + C::OFF_ROWS + C::ROWS, p.dsum + row_base + q0, C::ROWS, qf);
    nqi = i + 1;
  }
  // Drain, always: every copy this thread started lands before the CTA exits.
  wait_bar_drain(bk, 0, ctl);
  wait_bar_drain(bv, 0, ctl);
  if (nqi > 0) wait_bar_drain(qf, (nqi - 1) & 1, ctl);
  if (noi > 0) wait_bar_drain(of, (noi - 1) & 1, ctl);
}

// MMA warp: dP^T_0, then per Q tile i: S^T_i, dP^T_{i+1} (once the softmax has
// read dP^T_i), dK_i and dQ^T_i (once dS_i is written).
template <bool BF16>
__device__ __forceinline__ void dkdq_mma(uint32_t base, uint32_t tmem, int nq, const DCtl& ctl) {
  using C = CB;
  constexpr uint32_t fmt = BF16 ? 1u : 0u;
  constexpr uint32_t idesc_st = make_idesc(fmt, 0, 0, 128, C::BQ);  // S^T, dP^T: M = keys, N = queries
  constexpr uint32_t idesc_dk = make_idesc(fmt, 0, 1, 128, C::D);   // dK: A = dS^T, B = Q with d contiguous
  constexpr uint32_t idesc_dq = make_idesc(fmt, 1, 1, 128, C::BQ);  // dQ^T: A = K read d-major, B = dS^T
  const uint32_t b_done = dbar<C>(base, C::B_DONE), b_drain = dbar<C>(base, C::B_DRAIN);
  auto issue_dp = [&]() {
    mma_kmajor_d256(tmem + C::T_DP, base + C::OFF_V, C::KBLK, base + C::OFF_DO, C::QBLK, idesc_st);
    tc_commit_elect(dbar<C>(base, C::B_DPF));
    tc_commit_elect(dbar<C>(base, C::B_OE));  // dO_i is free
  };
  if (nq == 0) goto drain;
  if (!wait_bar_warp(dbar<C>(base, C::B_V), 0, ctl, kWhereBwdKV)) goto drain;
  if (!wait_bar_warp(dbar<C>(base, C::B_OF), 0, ctl, kWhereBwdDoFull)) goto drain;
  tc_fence_after();
  issue_dp();
  if (!wait_bar_warp(dbar<C>(base, C::B_K), 0, ctl, kWhereBwdKV)) goto drain;
  for (int i = 0; i < nq; ++i) {
    // S^T_i (its columns were read by the softmax of tile i-1, waited for below)
    if (!wait_bar_warp(dbar<C>(base, C::B_QF), i & 1, ctl, kWhereBwdQFull)) goto drain;
    tc_fence_after();
    mma_kmajor_d256(tmem + C::T_S, base + C::OFF_K, C::KBLK, base + C::OFF_Q, C::QBLK, idesc_st);
    tc_commit_elect(dbar<C>(base, C::B_SF));
    // dP^T_{i+1}, over dP^T_i, once the softmax has read S^T_i and dP^T_i
    if (!wait_bar_warp(dbar<C>(base, C::B_SC), i & 1, ctl, kWhereBwdDpFull)) goto drain;
    if (i + 1 < nq) {
      if (!wait_bar_warp(dbar<C>(base, C::B_OF), (i + 1) & 1, ctl, kWhereBwdDoFull)) goto drain;
      tc_fence_after();
      issue_dp();
    }
    // dK += dS^T_i Q_i (4 k-steps of 16 queries; Q's 16 rows are 2048 bytes,
    // its four 64-wide d blocks 8 KB apart)
    if (!wait_bar_warp(dbar<C>(base, C::B_DSF), i & 1, ctl, kWhereBwdDsFull)) goto drain;
    tc_fence_after();
    {
      const uint64_t a0 = opaque_d(smem_desc_sw128(base + C::OFF_DS, 16, 1024));
      const uint64_t b0 = opaque_d(smem_desc_sw128(base + C::OFF_Q, C::QBLK, 1024));
#pragma unroll
      for (int kk = 0; kk < C::BQ / 16; ++kk)
        mma_f16_ss_elect(tmem + C::T_DK, a0 + ((kk * 32u) >> 4), b0 + ((kk * 2048u) >> 4), idesc_dk,
                         (i > 0 || kk > 0) ? 1u : 0u);
    }
    tc_commit_elect(dbar<C>(base, C::B_QE));  // Q_i and its rows are free
    // dQ^T_i = K^T dS^T_i in two halves of d (8 k-steps of 16 keys each), over
    // dQ^T_{i-1} once the dQ warps have read it.
    if (i > 0 && !wait_bar_warp(dbar<C>(base, C::B_DQE), (i - 1) & 1, ctl, kWhereBwdDqEmpty)) goto drain;
    tc_fence_after();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint64_t a0 = opaque_d(smem_desc_sw128(base + C::OFF_K + 2 * h * C::KBLK, C::KBLK, 1024));
      const uint64_t b0 = opaque_d(smem_desc_sw128(base + C::OFF_DS, 1024, 1024));
#pragma unroll
      for (int kk = 0; kk < C::BK / 16; ++kk)
        mma_f16_ss_elect(tmem + C::T_DQ + 64 * h, a0 + ((kk * 2048u) >> 4), b0 + ((kk * 2048u) >> 4), idesc_dq,
                         kk > 0 ? 1u : 0u);
    }
    tc_commit_elect(dbar<C>(base, C::B_DQF));
    tc_commit_elect(dbar<C>(base, C::B_DSE));  // dK_i and dQ^T_i have read dS^T_i
  }
  tc_commit_elect(b_done);
drain:
  tc_commit_elect(b_drain);
  __all_sync(0xffffffffu, wait_bar_drain(b_drain, 0, ctl));
}

// Softmax warps 0-3 (thread = key): P from S^T_i, dS^T_i into shared memory;
// at the end dK.
template <bool BF16>
__device__ __forceinline__ void dkdq_softmax(const BwdParams& p, uint8_t* smem, uint32_t base, uint32_t tmem,
                                             const KeyTile& kt, const DCtl& ctl) {
  using C = CB;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const uint32_t lane_base = static_cast<uint32_t>(t & ~31) << 16;
  const uint32_t t_s = tmem + lane_base + C::T_S, t_dp = tmem + lane_base + C::T_DP;
  const float c = p.scale * kLog2eD;
  const float* lse2 = reinterpret_cast<const float*>(smem + C::OFF_ROWS);
  const float4* dsum4 = reinterpret_cast<const float4*>(smem + C::OFF_ROWS + C::ROWS);
  // Row t of dS^T (128-byte swizzle: 16-byte chunk k sits at k ^ (t & 7)).
  uint4* ds_row = reinterpret_cast<uint4*>(smem + C::OFF_DS + t * C::ROW);
  bool ok = true;
  for (int i = 0; i < kt.nq; ++i) {
    const int qt = kt.q_first + i;
    if (!named_bar_and(1, 128, wait_bar(dbar<C>(base, C::B_SF), i & 1, ctl, kWhereBwdSFull))) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t rs[2][32];
    tmem_ld32(t_s, rs[0]);
    tmem_ld32(t_s + 32, rs[1]);
    tmem_ld_wait();
    reg_fence(rs[0]);
    reg_fence(rs[1]);
    float ps[64];  // P * scale of this thread's key for the 64 queries of tile i
    uint32_t pk_unused[32];
    if (tile_masked(p, kt, qt))
      p_row<BF16, true, true>(rs, lse2, c, p.scale, mask_limit(p, kt, t, qt), pk_unused, ps);
    else
      p_row<BF16, false, true>(rs, lse2, c, p.scale, 0, pk_unused, ps);
    if (!named_bar_and(1, 128, wait_bar(dbar<C>(base, C::B_DPF), i & 1, ctl, kWhereBwdDpFull))) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t rdp[2][32];
    tmem_ld32(t_dp, rdp[0]);
    tmem_ld32(t_dp + 32, rdp[1]);
    tmem_ld_wait();
    reg_fence(rdp[0]);
    reg_fence(rdp[1]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(dbar<C>(base, C::B_SC));  // S^T_i and dP^T_i are in registers
    // dS^T_{i-1} has been read by dK_{i-1} and dQ^T_{i-1}.
    if (i > 0 && !named_bar_and(1, 128, wait_bar(dbar<C>(base, C::B_DSE), (i - 1) & 1, ctl, kWhereBwdDsEmpty))) {
      ok = false;
      break;
    }
    // dS^T * scale = P * scale * (dP^T - D), queries 8k..8k+7 in 16-byte chunk k.
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
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(dbar<C>(base, C::B_DSF));
  }
  if (ok && kt.nq > 0) ok = wait_bar(dbar<C>(base, C::B_DONE), 0, ctl, kWhereBwdDone);
  if (!named_bar_and(1, 128, ok)) return;
  tc_fence_after();
  // Every MMA is complete: the K tile's shared memory stages dK (the scale is already in dS).
  store_acc256<BF16>(tmem + lane_base + C::T_DK, base + C::OFF_K, t, 1, &p.tm_dk, kt.kv0, kt.bh);
}

// dQ warps 4-7 (thread = column 32w + lane of each half of d): dQ^T_i from
// TMEM, then one fp32 reduction per element into the accumulator.
__device__ __forceinline__ void dkdq_dq(const BwdParams& p, uint32_t base, uint32_t tmem, const KeyTile& kt,
                                        const DCtl& ctl) {
  using C = CB;
  const int t = threadIdx.x - 128;
  const int lane = t & 31, w = t >> 5;
  const uint32_t t_dq = tmem + (static_cast<uint32_t>(32 * w) << 16) + C::T_DQ;
  for (int i = 0; i < kt.nq; ++i) {
    if (!named_bar_and(2, 128, wait_bar(dbar<C>(base, C::B_DQF), i & 1, ctl, kWhereBwdDqFull))) break;
    tc_fence_after();
    uint32_t r[4][32];  // [half][query group of 32]
#pragma unroll
    for (int g = 0; g < 4; ++g) tmem_ld32(t_dq + 32 * g, r[g]);
    tmem_ld_wait();
#pragma unroll
    for (int g = 0; g < 4; ++g) reg_fence(r[g]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(dbar<C>(base, C::B_DQE));  // the MMA warp may reuse the columns
    const int q0 = (kt.q_first + i) * C::BQ;
    const int rows = min(C::BQ, p.N - q0);
    float* acc = p.dq_acc + (static_cast<size_t>(kt.bh) * p.N + q0) * C::D + 32 * w + lane;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int c = 0; c < C::BQ; ++c)
        if (c < rows) atomicAdd(acc + static_cast<size_t>(c) * C::D + 128 * h, __uint_as_float(r[2 * h + c / 32][c % 32]));
  }
}

template <bool BF16>
__global__ void __launch_bounds__(CB::THREADS, 1) fa_bwd_dkdq256_kernel(const __grid_constant__ BwdParams p) {
  using C = CB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5;
  const KeyTile kt = key_tile(p);
  if (kt.nq == 0) {
    // Every key of this tile is masked: its dK rows are zero and it adds nothing to dQ.
    zero_key_rows(p, p.dk, kt, C::THREADS);
    return;
  }
  if (threadIdx.x == 0) {
    const int one[] = {C::B_K, C::B_V, C::B_QF, C::B_QE, C::B_OF, C::B_OE, C::B_SF, C::B_DPF,
                       C::B_DSE, C::B_DQF, C::B_DONE, C::B_DRAIN};
    for (int b : one) mbar_init(dbar<C>(base, b), 1);
    mbar_init(dbar<C>(base, C::B_SC), 4);   // one arrival per softmax warp
    mbar_init(dbar<C>(base, C::B_DSF), 4);  // one arrival per softmax warp
    mbar_init(dbar<C>(base, C::B_DQE), 4);  // one arrival per dQ warp
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
  const DCtl ctl{p, base + C::OFF_MISC + 4};
  if (warp == C::WARP_TMA) {
    if ((threadIdx.x & 31) == 0) dkdq_producer(p, base, kt, ctl);
    __syncwarp();
  } else if (warp == C::WARP_MMA) {
    dkdq_mma<BF16>(base, tmem, kt.nq, ctl);
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    dkdq_dq(p, base, tmem, kt, ctl);
  } else if (warp < 4) {
    dkdq_softmax<BF16>(p, smem, base, tmem, kt, ctl);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// The dynamic shared memory attribute of one kernel, set once per device
// (C and BF16 name the kernel: one static flag word per instantiation).
template <class C, bool BF16, class K>
cudaError_t set_smem_once(K kern) {
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
  return cudaSuccess;
}

template <bool BF16>
cudaError_t launch_main256(const BwdParams& p, cudaStream_t stream) {
  auto ka = fa_bwd_dv256_kernel<BF16>;
  auto kb = fa_bwd_dkdq256_kernel<BF16>;
  cudaError_t e = set_smem_once<CA, BF16>(ka);
  if (e != cudaSuccess) return e;
  e = set_smem_once<CB, BF16>(kb);
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>(p.B) * p.H * ((p.N + B256::BK - 1) / B256::BK);
  if (ctas <= 0 || ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  ka<<<dim3(static_cast<unsigned>(ctas)), dim3(CA::THREADS), CA::SMEM_BYTES, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kb<<<dim3(static_cast<unsigned>(ctas)), dim3(CB::THREADS), CB::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_d256(const BwdParams& p, bool bf16, cudaStream_t stream) {
  return bf16 ? launch_main256<true>(p, stream) : launch_main256<false>(p, stream);
}

}  // namespace fa
