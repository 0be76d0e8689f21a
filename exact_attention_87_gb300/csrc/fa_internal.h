// fa_internal.h — parameter block and launch entry points shared by the host
// API (fa_api.cu) and the kernel translation units. Not part of the C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Bits of the device status word.
enum : unsigned int {
  kStatusTimeout = 1u,    // some wait gave up
  kStatusSmemAlign = 2u,  // a kernel found its dynamic shared memory misaligned and did nothing
};
// Where a wait gave up (stored in bits 8-15 of the status word, first writer wins).
enum : unsigned int {
  kWhereQ = 1, kWhereKEmpty, kWhereVEmpty, kWhereKFull, kWhereVFull, kWhereSFull, kWherePFull,
  kWhereODone, kWhereDrain, kWhereF32Mma, kWhereTurn,
  // backward kernel
  kWhereBwdKV, kWhereBwdQFull, kWhereBwdQEmpty, kWhereBwdDoFull, kWhereBwdDoEmpty, kWhereBwdSFull,
  kWhereBwdDpFull, kWhereBwdPFull, kWhereBwdDsFull, kWhereBwdDsEmpty, kWhereBwdDqFull, kWhereBwdDqEmpty,
  kWhereBwdDone
};

// Everything a forward kernel needs; passed by value as a __grid_constant__.
struct alignas(64) FwdParams {
  CUtensorMap tm_q;  // [B*H, N, d] boxes of 64 x 128 (16-bit path)
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  unsigned int* status;     // device status word of this module on this device
  long long wait_limit;     // clock64 cycles a barrier wait may spin before giving up
  int B, H, N, d;
  float scale;
  int num_sms;
  // Split-KV: each CTA covers split_tiles K/V tiles of one of num_splits key
  // ranges and writes its normalised fp32 O and its LSE to o_part / lse_part
  // ([num_splits, R, d] and [num_splits, R] over the R = B*H*N - merge_row0
  // rows from merge_row0 on); num_splits == 1: no split.
  int num_splits;
  int split_tiles;
  float* o_part;
  float* lse_part;
  // Keys: K and V hold Nk rows (Nk = N except for fa_fwd_partial). partial = 1:
  // the 16-bit kernel writes its normalised fp32 O and LSE to o_part / lse_part
  // as the one part of a merge done elsewhere (fa_merge).
  int Nk;
  int partial;
  // Work units of this launch of the 16-bit kernel: Q blocks [qunit0,
  // qunit0 + qunit_count) of the B*H*ceil(N/q) in (b*h, block) order (q =
  // fwd_q_block(d)), each split num_splits ways (qunit_count = 0: all of them). The split-KV merge
  // covers rows [merge_row0, B*H*N). The wave tail of a launch is split this
  // way: full waves unsplit, the last partial wave's units split.
  int qunit0;
  int qunit_count;
  long long merge_row0;
  // Masks: causal (row i sees keys j <= i) and per-batch key lengths
  // (klen[b]: keys j >= klen[b] masked; NULL = all N keys).
  int causal;
  const int* klen;
  // Streamed tail of the persistent d = 128 form (st_ctas > 0; unmasked, no
  // split): units before st_unit0 are handed out whole, round by round; the
  // K/V tiles of units [st_unit0, units) are laid end to end (st_tiles in
  // all) and CTA c < st_ctas takes the range [st_begin(c), st_begin(c + 1)).
  // Units a range boundary cuts are computed in pieces: normalised fp32 O
  // and LSE of each piece go to a slot of o_part / lse_part ([2 st_ctas, 256,
  // d] and [2 st_ctas, 256]) and a merge pass combines them.
  int st_unit0;
  int st_tiles;
  int st_ctas;
  // Host side only: launch this kernel as a programmatic dependent of the
  // previous kernel in the stream (it may start while that kernel's last
  // CTAs run; it reads none of its results, and its CTAs wait for that
  // kernel's completion before they exit, so that the stream's order of
  // completion is kept).
  int launch_pdl;
  // Used only by the testing build (-DFA_TESTING); zero / NULL otherwise.
  int inject;                       // 1: the producer skips the V load of tile 0
  float* stats_trace;               // [B*H*N, nkv, 2]: (m in natural-log units, l) after each K/V tile
  unsigned long long* timeline;     // [kTraceCtas, kTraceEvents, kTraceTiles] clock64 stamps
  float rescale_tau;                // lazy-rescale threshold (log2 units); the product build uses 15
};

// Everything the backward kernels need; passed by value as a __grid_constant__.
struct alignas(64) BwdParams {
  CUtensorMap tm_q;      // [B*H, N, d] 16-bit, boxes of 64 x 128 rows
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  CUtensorMap tm_dk;
  CUtensorMap tm_dv;
  CUtensorMap tm_dqacc;  // [B*H, N, d] fp32, boxes of 32 x 128 rows (reduce-add target)
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  float* dq_acc;         // workspace: fp32 dQ accumulator [B*H, N, d]
  float* lse2;           // workspace: LSE * log2(e) per row, [B*H, n_pad]; +inf on padding rows
  float* dsum;           // workspace: D_i = sum_c dO_ic O_ic per row, [B*H, n_pad]; 0 on padding rows
  unsigned int* status;
  long long wait_limit;
  int B, H, N, d;
  int n_pad;             // N rounded up to the 128-row tile
  float scale;
  // Used only by the testing build (-DFA_TESTING); zero / NULL otherwise.
  int inject;                    // 1: the producer skips the dO load of Q tile 0
  unsigned long long* timeline;  // [kTraceCtas, kTraceEvents, kTraceTiles] clock64 stamps
  // Masks (as FwdParams): causal (row i sees keys j <= i) and per-batch key
  // lengths (klen[b]: keys j >= klen[b] masked; NULL = all N keys). dK and dV
  // rows of fully masked key tiles are written as zeros through dk / dv.
  int causal;
  const int* klen;
  void* dk;
  void* dv;
};

// Lazy-rescale threshold of the 16-bit kernels in log2 units: P, taken
// against a row's reference max, stays <= 2^15 (fits fp16, whose largest
// value is 65504, and bf16), so the reference trails the running max by at
// most 15. The testing build can override it per call (FwdParams::rescale_tau).
constexpr float kRescaleThresholdLog2 = 15.0f;

// Tile sizes of the fp16/bf16 kernel: Q rows per sub-tile (two sub-tiles per
// CTA) and keys per K/V tile; the host encodes the TMA boxes with them.
constexpr int kF16BlockQ = 128, kF16BlockKV = 128;
// Tile sizes of the d = 256 kernel: Q rows per CTA (one Q tile) and keys per
// K/V tile (its K and V TMA boxes are this many rows).
constexpr int kD256BlockQ = 128, kD256BlockKV = 64;
// Rows of the K and V TMA boxes of the 16-bit forward kernel for head dimension d.
constexpr int fwd_kv_box_rows(int d) { return d == 256 ? kD256BlockKV : kF16BlockKV; }
// Q rows of one work unit of the 16-bit forward kernel for head dimension d
// (two 128-row sub-tiles for d = 64 / 128, one 128-row tile for d = 256).
constexpr int fwd_q_block(int d) { return d == 256 ? kD256BlockQ : 2 * kF16BlockQ; }

// Streamed tail (see FwdParams::st_ctas): first tail tile of CTA c's range
// (c = ctas: the end of the last range). Ranges are as equal as whole tiles
// allow; some are empty when the tail has fewer tiles than CTAs. 32-bit
// arithmetic: the host streams a tail only when tiles * ctas < 2^31.
__host__ __device__ inline int st_begin(int tiles, int ctas, int c) { return c * tiles / ctas; }
// One piece of CTA c's range: its q-th (0: the one holding the range's first
// tile), in tail unit i (counted from st_unit0), tiles [t0, t1) of the n in a
// unit; slot < 0 when the piece is the whole unit (written out directly),
// else 2c for the range's first piece and 2c + 1 for its last.
struct StPiece {
  int i, t0, t1, slot;
};
__host__ __device__ inline bool st_piece(int tiles, int ctas, int n, int c, int q, StPiece& pc) {
  const int a = st_begin(tiles, ctas, c), b = st_begin(tiles, ctas, c + 1);
  const int x = q == 0 ? a : (a / n + q) * n;
  if (q < 0 || x >= b) return false;
  pc.i = x / n;
  pc.t0 = x - pc.i * n;
  pc.t1 = b - x < n - pc.t0 ? pc.t0 + (b - x) : n;
  pc.slot = (pc.t0 == 0 && pc.t1 == n) ? -1 : 2 * c + (q == 0 ? 0 : 1);
  return true;
}
// The CTAs whose ranges hold tiles of tail unit i: c_lo .. c_hi (one CTA: the
// unit is whole in it). A CTA c in between with an empty range has no piece;
// the others' pieces sit in slot 2c when the range starts inside the unit,
// 2c + 1 when it started in an earlier one.
__host__ __device__ inline void st_unit_ctas(int tiles, int ctas, int n, int i, int& c_lo, int& c_hi) {
  const int x = i * n, e = x + n;
  c_lo = ((x + 1) * ctas - 1) / tiles;
  c_hi = (e * ctas - 1) / tiles;
}

// Timeline trace layout of the testing build.
constexpr int kTraceCtas = 8, kTraceTiles = 64, kTraceEvents = 32;
enum : int {
  kEvS0Issued = 0, kEvS1Issued, kEvPV0Issued, kEvPV1Issued, kEvSm0SFull, kEvSm0PArrive, kEvSm1SFull,
  kEvSm1PArrive, kEvKIssued, kEvVIssued, kEvMmaKFull, kEvMmaVFull, kEvCta
};
// Backward kernel events (tile index = Q tile i): MMA issue of dV_i, dP_i,
// S_{i+1}, dK_i, dQ_i; softmax warpgroup 0 (thread 0): S_i ready, P_i
// arrived, dQ_i ready, dQ_i reduce-adds issued, dP_i ready, dS_i arrived,
// dS^T half free (reduce-adds of dQ_{i-1} have read it), dQ_i out of TMEM;
// warpgroup 1: P_i and dS_i arrived.
// Then, for the MMA warp, the moment each product's waits are over (before
// its first MMA), and the producer's issue of the Q_i and dO_i loads.
enum : int {
  kBvDV = 0, kBvDP, kBvS, kBvDK, kBvDQ, kBvSmS, kBvSmP, kBvSmDq, kBvSmRed, kBvSmDp, kBvSmDs, kBvSmDsFree,
  kBvSmDqLoaded, kBvCta, kBvW1P, kBvW1Ds, kBvDVReady, kBvDPReady, kBvSReady, kBvDKReady, kBvDQReady, kBvQLoad,
  kBvDOLoad, kBvSmPChunk0, kBvSmDsWaited, kBvSmDsChunk0, kBvSmDsChunk1
};

// Launch the 16-bit (fp16 / bf16) forward kernel for head dimension p.d (64 or 128).
cudaError_t launch_fwd_f16(const FwdParams& p, bool bf16, cudaStream_t stream);
// Merge num_splits parts in o_part / lse_part (rows from merge_row0 on) into
// O (dtype of the 16-bit path, head dimension 64, 128 or 256) and LSE; rows
// with no key in any part get O = 0, LSE = -inf. Serves split-KV and fa_merge
// alike.
cudaError_t launch_merge(const FwdParams& p, bool bf16, cudaStream_t stream);
// Whether the persistent d = 128 forward takes this launch (also the
// condition for a streamed tail, st_ctas > 0).
bool fwd_persist_eligible(const FwdParams& p);
// Backward: row statistics (D, LSE * log2 e) and a zeroed dQ accumulator;
// the main dK/dV/dQ kernel; the dQ accumulator rounded into dQ.
// Head dimension 64, 128 or 256 (the last through launch_bwd_main_d256).
cudaError_t launch_bwd_f16(const BwdParams& p, bool bf16, cudaStream_t stream);
// The two main kernels of the d = 256 backward (dV; then dK and the dQ
// contributions), between the row statistics and the dQ rounding.
cudaError_t launch_bwd_main_d256(const BwdParams& p, bool bf16, cudaStream_t stream);
// Launch the 16-bit forward kernel for head dimension 256 (same parameter
// block and work-unit scheme as launch_fwd_f16, with 128-row Q tiles and
// 64-key K/V tiles).
cudaError_t launch_fwd_d256(const FwdParams& p, bool bf16, cudaStream_t stream);
// Launch the fp32 (3 x TF32) forward kernel.
cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream);

}  // namespace fa
