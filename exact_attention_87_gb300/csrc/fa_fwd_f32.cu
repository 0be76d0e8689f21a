// fa_fwd_f32.cu — FlashAttention forward for fp32 inputs on sm_103a.
//
// Same recurrence as the 16-bit kernel (MUSA SDK guide, "FlashAttention 优化",
// "FlashAttention 完整算法" steps 1-4), here with the eager per-tile rescale
// of the formula (step 3e: O <- diag(exp(m_old - m_new)) O + P V).
//
// Precision: the accuracy target for fp32 inputs (max |err| < 1e-5, the
// dataflow page's section 4.1) rules out a single TF32 product (about 1e-3
// error). Each product X.Y therefore runs as three TF32 tensor-core products
// hi(X)hi(Y) + hi(X)lo(Y) + lo(X)hi(Y) with fp32 accumulation in TMEM, where
// hi(x) keeps the sign, exponent and top 10 mantissa bits of x (exactly
// representable in TF32) and lo(x) = x - hi(x) (exact in fp32). The dropped
// lo*lo term and the TF32 rounding of lo are about 2^-22 relative.
//
// Mapping: one CTA per (batch*head, 128-row Q tile), one warpgroup (thread =
// row = TMEM lane). Q hi/lo stay resident in shared memory; each K/V tile is
// loaded with coalesced 16-byte loads, split, and written in the 128-byte
// swizzled layout the MMA descriptors expect (V transposed, so that every
// operand is K-major); P hi/lo go through shared memory. One thread issues the MMAs; completion is signalled through mbarriers
// by tcgen05.commit. This path targets small, latency-bound fp32 problems.
#include <atomic>

#include "fa_device_common.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg32 {
  static constexpr int BM = 128;
  static constexpr int BN = (D == 128) ? 32 : 64;   // keys per tile (shared memory bound)
  static constexpr uint32_t Q_BYTES = BM * D * 4;    // one of Q_hi / Q_lo
  static constexpr uint32_t KV_BYTES = BN * D * 4;   // one of K_hi / K_lo / V_hi / V_lo
  static constexpr uint32_t P_BYTES = BM * BN * 4;   // one of P_hi / P_lo
  static constexpr uint32_t OFF_QH = 0, OFF_QL = OFF_QH + Q_BYTES;
  static constexpr uint32_t OFF_KH = OFF_QL + Q_BYTES, OFF_KL = OFF_KH + KV_BYTES;
  static constexpr uint32_t OFF_VH = OFF_KL + KV_BYTES, OFF_VL = OFF_VH + KV_BYTES;
  static constexpr uint32_t OFF_PH = OFF_VL + KV_BYTES, OFF_PL = OFF_PH + P_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_PL + P_BYTES;  // bar_s, bar_o, bar_drain
  static constexpr uint32_t OFF_MISC = OFF_BAR + 3 * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr uint32_t T_S = 0, T_O = 128;
  static constexpr int THREADS = 128;
};

__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// Byte offset of element (r, k) of a K-major (or MN-major) 32-bit operand
// stored as column blocks of 32 elements, each block `rows` x 128 bytes with
// the 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t sw128_off32(uint32_t r, uint32_t k, uint32_t rows) {
  const uint32_t blk = k >> 5, kin = k & 31u;
  const uint32_t chunk = (kin >> 2) ^ (r & 7u);
  return blk * rows * 128u + r * 128u + chunk * 16u + (kin & 3u) * 4u;
}

// Load rows [row0, row0 + rows) of a [N, D] fp32 matrix (rows >= N read as 0),
// split each value into hi/lo, and store both in the swizzled layout.
template <int D>
__device__ __forceinline__ void load_split(const float* __restrict__ g, int row0, int rows, int N, uint32_t s_hi,
                                           uint32_t s_lo) {
  constexpr int V4_PER_ROW = D / 4;
  const int total = rows * V4_PER_ROW;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int r = idx / V4_PER_ROW, c4 = idx % V4_PER_ROW;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + r < N) x = __ldg(reinterpret_cast<const float4*>(g + static_cast<size_t>(row0 + r) * D) + c4);
    const float4 h = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
    const float4 l = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
    const uint32_t off = sw128_off32(r, c4 * 4, rows);  // 4 consecutive columns share one 16-byte chunk
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(s_hi + off), "f"(h.x), "f"(h.y), "f"(h.z),
                 "f"(h.w)
                 : "memory");
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(s_lo + off), "f"(l.x), "f"(l.y), "f"(l.z),
                 "f"(l.w)
                 : "memory");
  }
}

// Same for a [N, D] matrix V, stored transposed: element (key j, column n) at
// row n, K index j - row0, so that V is a K-major B operand ([D rows] x [BN keys]).
template <int D, int BN>
__device__ __forceinline__ void load_split_t(const float* __restrict__ g, int row0, int N, uint32_t s_hi,
                                             uint32_t s_lo) {
  constexpr int V4_PER_ROW = D / 4;
  for (int idx = threadIdx.x; idx < BN * V4_PER_ROW; idx += blockDim.x) {
    const int r = idx / V4_PER_ROW, c4 = idx % V4_PER_ROW;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + r < N) x = __ldg(reinterpret_cast<const float4*>(g + static_cast<size_t>(row0 + r) * D) + c4);
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float h = tf32_hi(xs[e]);
      const uint32_t off = sw128_off32(c4 * 4 + e, r, D);
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(s_hi + off), "f"(h) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(s_lo + off), "f"(xs[e] - h) : "memory");
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128, 1) fa_fwd_f32_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg32<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem_raw + (base - raw) + C::OFF_MISC);
  const uint32_t bar_s = base + C::OFF_BAR, bar_o = bar_s + 8, bar_drain = bar_s + 16;

  const int t = threadIdx.x, warp = t >> 5;
  const int nqb = (p.N + C::BM - 1) / C::BM;
  const int bh = blockIdx.x / nqb;
  const int row0 = (blockIdx.x % nqb) * C::BM;
  // Keys this tile may see: [0, key_end); causal rows see keys up to themselves.
  const int key_end = p.klen ? max(0, min(p.N, p.klen[bh / p.H])) : p.N;
  const int tile_end = p.causal ? min(key_end, row0 + C::BM) : key_end;
  const int nkv = (tile_end + C::BN - 1) / C::BN;
  const size_t head = static_cast<size_t>(bh) * p.N * D;
  const float* q = static_cast<const float*>(p.q) + head;
  const float* k = static_cast<const float*>(p.k) + head;
  const float* v = static_cast<const float*>(p.v) + head;

  if (t == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_drain, 1);
    misc[1] = 0;
    mbar_init_fence();
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(base + C::OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  load_split<D>(q, row0, C::BM, p.N, base + C::OFF_QH, base + C::OFF_QL);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const WaitCtl ctl{p, base + C::OFF_MISC + 4};  // misc[1] is the abort flag
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t t_s = tmem + lane_base + C::T_S, t_o = tmem + lane_base + C::T_O;

  constexpr uint32_t idesc_s = make_idesc(2, 0, 0, 128, C::BN);  // tf32, Q and K K-major
  constexpr uint32_t idesc_o = make_idesc(2, 0, 0, 128, D);      // tf32, P and V^T both K-major
  const float c = p.scale * kLog2e;
  float m = -INFINITY, l = 0.f;
  bool ok = true;

  for (int j = 0; j < nkv && ok; ++j) {
    load_split<D>(k, j * C::BN, C::BN, p.N, base + C::OFF_KH, base + C::OFF_KL);
    load_split_t<D, C::BN>(v, j * C::BN, p.N, base + C::OFF_VH, base + C::OFF_VL);
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      // S = Qh Kh^T + Qh Kl^T + Ql Kh^T; each MMA covers 8 of the d columns.
#pragma unroll
      for (int kk = 0; kk < D / 8; ++kk) {
        const uint32_t off = (kk & 3) * 32u;  // 8 tf32 elements = 32 bytes inside the swizzled row
        const uint32_t qblk = (kk / 4) * C::BM * 128u, kblk = (kk / 4) * C::BN * 128u;
        const uint64_t qh = smem_desc_sw128(base + C::OFF_QH + qblk + off, 16, 1024);
        const uint64_t ql = smem_desc_sw128(base + C::OFF_QL + qblk + off, 16, 1024);
        const uint64_t kh = smem_desc_sw128(base + C::OFF_KH + kblk + off, 16, 1024);
        const uint64_t kl = smem_desc_sw128(base + C::OFF_KL + kblk + off, 16, 1024);
        mma_tf32_ss_elect(tmem + C::T_S, qh, kh, idesc_s, kk > 0 ? 1u : 0u);
        mma_tf32_ss_elect(tmem + C::T_S, qh, kl, idesc_s, 1u);
        mma_tf32_ss_elect(tmem + C::T_S, ql, kh, idesc_s, 1u);
      }
      tc_commit_elect(bar_s);
    }
    __syncwarp();
    // CTA-uniform outcome: every thread takes the same path through the barriers below.
    if (!__syncthreads_and(wait_bar(bar_s, j & 1, ctl, kWhereF32Mma))) { ok = false; break; }
    tc_fence_after();

    uint32_t sr[C::BN];
#pragma unroll
    for (int qd = 0; qd < C::BN / 32; ++qd)
      tmem_ld32(t_s + 32 * qd, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * qd]));
    tmem_ld_wait();
#pragma unroll
    for (int qd = 0; qd < C::BN / 32; ++qd) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&sr[32 * qd]));
    const int my_row = row0 + t;
    const int valid = (p.causal ? min(key_end, my_row + 1) : key_end) - j * C::BN;
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < C::BN; ++u) {
      if (u >= valid) sr[u] = __float_as_uint(-INFINITY);
      mx = fmaxf(mx, __uint_as_float(sr[u]));
    }
    const float m_new = fmaxf(m, mx * c);
    const float alpha = (j == 0) ? 0.f : ex2_approx(m - m_new);
    m = m_new;
    float rs = 0.f;
#pragma unroll
    for (int u = 0; u < C::BN; u += 4) {
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pv[e] = ex2_approx(fmaf(__uint_as_float(sr[u + e]), c, -m));
        rs += pv[e];
      }
      const uint32_t off = sw128_off32(t, u, C::BM);
      const float h0 = tf32_hi(pv[0]), h1 = tf32_hi(pv[1]), h2 = tf32_hi(pv[2]), h3 = tf32_hi(pv[3]);
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(base + C::OFF_PH + off), "f"(h0), "f"(h1),
                   "f"(h2), "f"(h3)
                   : "memory");
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(base + C::OFF_PL + off), "f"(pv[0] - h0),
                   "f"(pv[1] - h1), "f"(pv[2] - h2), "f"(pv[3] - h3)
                   : "memory");
    }
    l = l * alpha + rs;
    if (j > 0) {
      // O <- alpha O before this tile's P.V (the previous P.V completed: bar_o was waited on).
#pragma unroll
      for (int qd = 0; qd < D / 32; ++qd) {
        uint32_t r[32];
        tmem_ld32(t_o + 32 * qd, r);
        tmem_ld_wait();
        reg_fence(r);
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * alpha);
        tmem_st32(t_o + 32 * qd, r);
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      // O += Ph Vh + Ph Vl + Pl Vh; each MMA covers 8 keys.
#pragma unroll
      for (int kk = 0; kk < C::BN / 8; ++kk) {
        const uint32_t koff = (kk & 3) * 32u;  // 8 keys = 32 bytes inside the swizzled row
        const uint32_t poff = (kk / 4) * C::BM * 128u + koff;
        const uint32_t voff = (kk / 4) * D * 128u + koff;
        const uint64_t ph = smem_desc_sw128(base + C::OFF_PH + poff, 16, 1024);
        const uint64_t pl = smem_desc_sw128(base + C::OFF_PL + poff, 16, 1024);
        const uint64_t vh = smem_desc_sw128(base + C::OFF_VH + voff, 16, 1024);
        const uint64_t vl = smem_desc_sw128(base + C::OFF_VL + voff, 16, 1024);
        mma_tf32_ss_elect(tmem + C::T_O, ph, vh, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        mma_tf32_ss_elect(tmem + C::T_O, ph, vl, idesc_o, 1u);
        mma_tf32_ss_elect(tmem + C::T_O, pl, vh, idesc_o, 1u);
      }
      tc_commit_elect(bar_o);
    }
    __syncwarp();
    // Shared K/V/P buffers are reused by the next tile only after this P.V is done.
    if (!__syncthreads_and(wait_bar(bar_o, j & 1, ctl, kWhereF32Mma))) { ok = false; break; }
    tc_fence_after();
  }

  if (ok) {
    // No key to attend to (key length 0): O = 0, LSE = -inf instead of 0/0.
    const bool empty = nkv == 0;
    const float inv_l = empty ? 0.f : 1.0f / l;
    const int row = row0 + t;
    float* o = static_cast<float*>(p.o) + head;
#pragma unroll
    for (int qd = 0; qd < D / 32; ++qd) {
      uint32_t r[32];
      tmem_ld32(t_o + 32 * qd, r);
      tmem_ld_wait();
      reg_fence(r);
      if (empty) {
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] = 0u;  // TMEM O was never written
      }
      if (row < p.N) {
        float4* dst = reinterpret_cast<float4*>(o + static_cast<size_t>(row) * D + 32 * qd);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          dst[u] = make_float4(__uint_as_float(r[4 * u]) * inv_l, __uint_as_float(r[4 * u + 1]) * inv_l,
                               __uint_as_float(r[4 * u + 2]) * inv_l, __uint_as_float(r[4 * u + 3]) * inv_l);
      }
    }
    if (row < p.N) p.lse[static_cast<size_t>(bh) * p.N + row] = empty ? -INFINITY : (m + lg2_approx(l)) * kLn2;
  } else if (warp == 0) {
    // Drain: every MMA this warp issued must finish before TMEM is freed.
    tc_commit_elect(bar_drain);
    __all_sync(0xffffffffu, wait_bar_drain(bar_drain, 0, ctl));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch32(const FwdParams& p, cudaStream_t stream) {
  using C = Cfg32<D>;
  static_assert(C::SMEM_BYTES <= 232448, "shared memory budget");
  auto kern = fa_fwd_f32_kernel<D>;
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit);
  }
  const long long units = static_cast<long long>(p.B) * p.H * ((p.N + C::BM - 1) / C::BM);
  if (units <= 0 || units > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<dim3(static_cast<unsigned>(units)), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream) {
  if (p.d == 128) return launch32<128>(p, stream);
  if (p.d == 64) return launch32<64>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
