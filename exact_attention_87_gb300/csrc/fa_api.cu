// fa_api.cu — host side of the C ABI declared in include/fa.h: argument
// validation, per-device checks, TMA descriptor encoding and kernel launch.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fa.h"
#ifdef FA_TESTING
#include "fa_testing.h"
#endif
#include "fa_internal.h"
#ifdef FA_TESTING
#include "fa_bwd_order.cuh"
#include "fa_fwd_order.cuh"
#endif

// Device status word of this module: [0] flags (kStatusTimeout), [1] where the
// first timeout happened. Kernels receive its address as a parameter.
__device__ unsigned int g_fa_status[2];

// Built-in scratch of fa_fwd_splitkv_noalloc (split-KV partial O and LSE).
// Host code must not pass this name to a kernel: it is a host-side stand-in;
// the device address comes from cudaGetSymbolAddress (noalloc_scratch()).
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool is_sm103 = false;
  int num_sms = 0;
  unsigned int* status = nullptr;
  void* noalloc_scratch = nullptr;  // device address of g_fa_noalloc_scratch (looked up on first use)
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
long long g_wait_limit = 0;

#ifdef FA_TESTING
// Testing build: when set, the entry points return FA_OK after every argument
// and device check, before anything is enqueued (so that argument-error tests
// can pass placeholder addresses: a check that regressed then shows up as a
// wrong status, never as a launch on memory that does not exist).
std::atomic<int> g_dry_run{0};
#define FA_DRY_RUN_RETURN() \
  do {                      \
    if (g_dry_run.load()) return FA_OK; \
  } while (0)
#else
#define FA_DRY_RUN_RETURN() \
  do {                      \
  } while (0)
#endif

long long wait_limit_cycles() {
  if (g_wait_limit == 0) {
    long long v = 1ll << 32;  // ~2 s at GB300 clocks
    if (const char* e = std::getenv("FA_WAIT_LIMIT_CYCLES")) {
      long long x = std::atoll(e);
      if (x > 0) v = x;
    }
    g_wait_limit = v;
  }
  return g_wait_limit;
}

// Per-device facts, probed once under the lock. Returns FA_OK / FA_ERR_ARCH / FA_ERR_CUDA.
int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    d.is_sm103 = (major == 10 && minor == 3);
    d.num_sms = sms;
    if (d.is_sm103) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
      d.status = static_cast<unsigned int*>(p);
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FA_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.probed = true;
  }
  *out = d;
  return d.is_sm103 ? FA_OK : FA_ERR_ARCH;
}

// [B*H, N, d] tensor of 16-bit elements, boxes of 64 (d) x `box_rows` rows, 128-byte swizzle.
bool encode_bhnd_16bit(CUtensorMap* map, const void* ptr, int BH, int N, int d, CUtensorMapDataType dt,
                       int box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [B*H, N, d] fp32 tensor, boxes of 32 (d) x 128 rows, 128-byte swizzle (the dQ accumulator).
bool encode_bhnd_f32_box32(CUtensorMap* map, void* ptr, int BH, int N, int d) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the built-in scratch on the current device, looked up once
// per device with that device current. Returns FA_OK / FA_ERR_CUDA / FA_ERR_ARCH.
int noalloc_scratch(void** out) {
  DeviceInfo dev;
  const int st = device_info(&dev);
  if (st != FA_OK) return st;
  int ord = 0;
  if (cudaGetDevice(&ord) != cudaSuccess) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[ord];
  if (!d.noalloc_scratch) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fa_noalloc_scratch) != cudaSuccess || ptr == nullptr) return FA_ERR_CUDA;
    d.noalloc_scratch = ptr;
  }
  *out = d.noalloc_scratch;
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_abi_version(void) { return 100; }

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_DTYPE: return "dtype must be FA_F32, FA_F16 or FA_BF16";
    case FA_ERR_SHAPE: return "B, H and N must be >= 1 and B*H*N*d must stay below 2^40 elements";
    case FA_ERR_HEADDIM:
      return "head dimension d must be 64 or 128 (or 256 for the fp16/bf16 forward pass)";
    case FA_ERR_ALIGN: return "Q, K, V and O must be 16-byte aligned and LSE 4-byte aligned";
    case FA_ERR_CUDA: return "a CUDA call failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a kernel timed out waiting on an internal pipeline barrier";
    case FA_ERR_ARCH: return "the current device is not sm_103 (GB300)";
    case FA_ERR_SCALE: return "scale must be finite and > 0";
    case FA_ERR_WORKSPACE: return "split-KV workspace is NULL, not 256-byte aligned or smaller than required";
    case FA_ERR_SCRATCH_LIMIT:
      return "this shape's split-KV workspace exceeds the library's 32 MiB built-in scratch "
             "(fa_fwd_splitkv_noalloc); use fa_fwd_splitkv with a caller workspace";
    case FA_ERR_UNSUPPORTED: return "this entry point does not take the given dtype (fa_bwd takes FA_F16 or FA_BF16)";
    case FA_ERR_DEVICE_SMEM: return "a kernel found its dynamic shared memory misaligned and did no work";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace {

// Split-KV sizing. Work units of the 16-bit forward kernels are
// fa::fwd_q_block(d) Q rows (256, or 128 at d = 256) x (a key range of whole
// K/V tiles of fa::fwd_kv_box_rows(d) keys: 128, or 64 at d = 256).
long long kv_tiles(int N, int d) {
  const int t = fa::fwd_kv_box_rows(d);
  return (static_cast<long long>(N) + t - 1) / t;
}
long long q_blocks(int N, int d) {
  const int q = fa::fwd_q_block(d);
  return (static_cast<long long>(N) + q - 1) / q;
}
// 128-row tiles of the backward kernels.
long long bwd_tiles(int N) { return (static_cast<long long>(N) + fa::kF16BlockKV - 1) / fa::kF16BlockKV; }

// Effective split count: explicit requests are clamped so that every range
// holds at least one tile; 0 picks the count with the smallest modelled time:
//   waves(s) * (tiles/s + 1) * t_tile            partial passes (+1 tile of set-up per unit)
// + (s > 1) * (2 * s * rows * d * 4 bytes / 5 TB/s + 5 us)   the merge pass
// with t_tile ~ 2 us * d / 128 for one 256-row unit and one 128-key tile on
// one SM (measured on GB300 at ~2 GHz), scaled by the unit's rows x keys for
// the d = 256 kernel's 128-row units and 64-key tiles (1 us).
// The tail plan: when the units end in a partial last wave, the full waves
// run unsplit and only the last wave's units are split (as many ways as fit
// in one wave), then merged:
//   W * (tiles + 1) * t_tile + (tiles/s + 1) * t_tile + merge of the tail rows
//   + b
// The last term is the launch boundary. The split tail is a programmatic
// dependent launch (its CTAs start as the full waves' CTAs finish); b = 5 us
// for d <= 128, and 20 us at d = 256, the boundary measured before the tail
// was launched that way (no measurement of d = 256 with it yet). Measured on
// GB300 with b = 20 us: with the tail split, B=1 H=8 N=16384 d=128 runs 8 %
// faster than unsplit (uniform 2-way splits 1 % slower) and B=4 H=16 N=4096
// d=256 (13.5 waves) 1 % slower (unsplit there).
struct SplitPlan {
  int splits;            // key ranges per split unit (1: unsplit)
  long long tail_qunit0; // >= 0: units before it unsplit, the rest split; < 0: every unit split alike
};

SplitPlan split_plan(int B, int H, int N, int d, int num_splits, int num_sms) {
  const long long tiles = kv_tiles(N, d);
  if (num_splits > 0) return {static_cast<int>(std::min<long long>(num_splits, tiles)), -1};
  const long long units = static_cast<long long>(B) * H * q_blocks(N, d);
  const double rows = static_cast<double>(B) * H * N;
  const double t_tile_us =
      2.0 * d / 128.0 * (fa::fwd_q_block(d) * fa::fwd_kv_box_rows(d)) / (2.0 * fa::kF16BlockQ * fa::kF16BlockKV);
  SplitPlan best{1, -1};
  double best_us = 1e300;
  for (int s = 1; s <= 16 && s <= tiles; ++s) {
    const long long per = (tiles + s - 1) / s;
    if ((tiles + per - 1) / per != s) continue;
    const double waves = static_cast<double>((units * s + num_sms - 1) / num_sms);
    double us = waves * (static_cast<double>(per) + 1.0) * t_tile_us;
    if (s > 1) us += 2.0 * s * rows * d * 4.0 / 5e12 * 1e6 + 5.0;
    if (us < best_us) { best_us = us; best = {s, -1}; }
  }
  const long long full = units / num_sms, tail = units - full * num_sms;
  if (full >= 1 && tail > 0) {
    const long long s = std::min<long long>({num_sms / tail, tiles, 16});
    if (s >= 2) {
      const long long per = (tiles + s - 1) / s;
      const double tail_rows = static_cast<double>(tail) * fa::fwd_q_block(d);
      const double us = static_cast<double>(full) * (static_cast<double>(tiles) + 1.0) * t_tile_us +
                        (static_cast<double>(per) + 1.0) * t_tile_us + 2.0 * s * tail_rows * d * 4.0 / 5e12 * 1e6 +
                        5.0 + (d == 256 ? 20.0 : 5.0);
      if (us < best_us) best = {static_cast<int>(s), full * num_sms};
    }
  }
  return best;
}

// Partial O and LSE of `splits` key ranges over the rows from row0 on (the
// rows of the split units: all rows, or those of the wave tail).
unsigned long long workspace_bytes_for(int B, int H, int N, int d, int splits, long long row0 = 0) {
  if (splits <= 1) return 0;
  const unsigned long long rows = (static_cast<unsigned long long>(B) * H * N - row0) * splits;
  const unsigned long long o_bytes = (rows * d * 4 + 255) & ~255ull;
  return o_bytes + rows * 4;
}

// First row of the split units of a plan (0 unless only the wave tail is split).
long long plan_row0(const SplitPlan& plan, int N, int d) {
  if (plan.tail_qunit0 <= 0) return 0;
  const long long nqb = q_blocks(N, d);
  return (plan.tail_qunit0 / nqb) * N + (plan.tail_qunit0 % nqb) * fa::fwd_q_block(d);
}

// Streamed tail of the persistent d = 128 forward (unmasked, N a multiple of
// 256 and at most 4096, where the persistent form runs; see
// fa::FwdParams::st_ctas): the full rounds of num_sms units run whole, the
// K/V tiles of the units left over are cut into one contiguous range per
// CTA, and the units a range boundary cuts are merged afterwards. Modelled
// time, in tiles of one 256-row unit and one 128-key tile on one SM
// (t_p ~ 1.63 us on GB300 in the persistent kernel):
//   whole units only:  ceil(units / num_sms) * n
//   streamed tail:     1.04 * (R * n + ceil(tail tiles / ctas) + 1)
//                      + (3 us + 2 * partial bytes / 4 TB/s) / t_p   (the merge)
// with R full rounds, n tiles per unit and `ctas` CTAs sharing the tail
// (num_sms / k for k = 1..8, at most kStreamMaxCtas so that the part slots
// fit the library's 32 MiB scratch); 1.04: the tile rate of the kernel
// instantiation that carries the tail's code (measured 2-5 % below the one
// without). The tail is streamed only when that saves at least two tiles.
// On B=8 H=12 N=2048 (768 units, 5.05 rounds) it takes 2-tile ranges on 76
// CTAs; on B=8 H=32 N=4096 (26.9 rounds) it does not pay.
struct StreamPlan {
  int unit0 = 0;            // first tail unit (R * num_sms)
  int tiles = 0;            // K/V tiles of the tail
  int ctas = 0;             // CTAs sharing the tail (0: no streamed tail)
  int max_pieces = 0;       // most pieces one unit is cut into
};
constexpr int kStreamRows = 2 * fa::kF16BlockQ;  // rows of a unit (and of a part slot)
constexpr unsigned long long stream_slot_bytes(int d) {
  return static_cast<unsigned long long>(kStreamRows) * (4ull * d + 4);
}
constexpr int kStreamMaxCtas = static_cast<int>(FA_NOALLOC_SCRATCH_BYTES / (2 * (stream_slot_bytes(128) + 512)));

unsigned long long stream_workspace_bytes(int ctas, int d) {
  if (ctas <= 0) return 0;
  const unsigned long long rows = 2ull * ctas * kStreamRows;
  return ((rows * d * 4 + 255) & ~255ull) + rows * 4;
}

StreamPlan stream_plan(int B, int H, int N, int d, int num_sms) {
  StreamPlan best;
  if (d != 128 || N % kStreamRows != 0 || N > 4096 || num_sms < 1) return best;
  const long long units = static_cast<long long>(B) * H * (N / kStreamRows);
  const int n = N / fa::kF16BlockKV;
  const long long R = units / num_sms, tail = units - R * num_sms;
  if (tail == 0 || units > 0x7fffffffLL) return best;
  const double t_p = 1.63;
  const long long T = tail * n;
  // 32-bit range arithmetic on the device
  if (T * num_sms >= (1ll << 31)) return best;
  double best_t = static_cast<double>(R + 1) * n - 2.0;
  int last = 0;
  for (int k = 1; k <= 8; ++k) {
    const int ctas = std::min((num_sms + k - 1) / k, kStreamMaxCtas);
    if (ctas == last || ctas < 1) continue;
    last = ctas;
    long long partial = 0;  // pieces written as parts: a range's first and last, when they cut a unit
    for (int c = 0; c < ctas; ++c) {
      const int a = fa::st_begin(static_cast<int>(T), ctas, c), b = fa::st_begin(static_cast<int>(T), ctas, c + 1);
      if (a == b) continue;
      fa::StPiece pc;
      fa::st_piece(static_cast<int>(T), ctas, n, c, 0, pc);
      if (pc.slot >= 0) ++partial;
      if (b > (a / n + 1) * n && b % n != 0) ++partial;
    }
    const double t = 1.04 * (static_cast<double>(R) * n + static_cast<double>((T + ctas - 1) / ctas) + 1.0) +
                     (3.0 + 2.0 * partial * stream_slot_bytes(d) / 4e12 * 1e6) / t_p;
    if (t < best_t) {
      best_t = t;
      best.unit0 = static_cast<int>(R * num_sms);
      best.tiles = static_cast<int>(T);
      best.ctas = ctas;
    }
  }
  if (best.ctas > 0) {
    for (int i = 0; i < tail; ++i) {
      int c_lo, c_hi, pieces = 0;
      fa::st_unit_ctas(best.tiles, best.ctas, n, i, c_lo, c_hi);
      for (int c = c_lo; c <= c_hi; ++c)
        if (fa::st_begin(best.tiles, best.ctas, c) != fa::st_begin(best.tiles, best.ctas, c + 1)) ++pieces;
      best.max_pieces = std::max(best.max_pieces, pieces);
    }
  }
  return best;
}

// What a 16-bit split-KV pass does for a shape on a device with num_sms SMs:
// the key ranges per split unit after clamping to whole tiles, the first
// split unit, the launches and the workspace. Host arithmetic only.
struct PlanSummary {
  int splits;              // key ranges of each split unit (1: nothing is split)
  long long first_split;   // first split work unit (all units: nothing is split)
  int launches;            // 1, 2 or 3
  unsigned long long workspace;
};

PlanSummary summarize_classic(int B, int H, int N, int d, int num_splits, int num_sms) {
  const long long units = static_cast<long long>(B) * H * q_blocks(N, d);
  const SplitPlan plan = split_plan(B, H, N, d, num_splits, num_sms);
  const long long tiles = kv_tiles(N, d);
  const long long per = (tiles + plan.splits - 1) / plan.splits;
  const int eff = static_cast<int>((tiles + per - 1) / per);
  if (eff <= 1) return {1, units, 1, 0};
  const bool tail = plan.tail_qunit0 > 0;
  return {eff, tail ? plan.tail_qunit0 : 0, tail ? 3 : 2,
          workspace_bytes_for(B, H, N, d, eff, tail ? plan_row0(plan, N, d) : 0)};
}

// The automatic count of an unmasked 16-bit call with d = 128 and N a
// multiple of 256 takes the streamed tail when it pays (2 launches: the
// persistent pass and the merge of the cut units; splits = the most pieces
// of one unit). Calls with masks take the key-range plan of the same
// arguments, so the workspace covers both.
PlanSummary summarize_plan(int B, int H, int N, int d, int num_splits, int num_sms) {
  const PlanSummary classic = summarize_classic(B, H, N, d, num_splits, num_sms);
  if (num_splits != 0) return classic;
  const StreamPlan sp = stream_plan(B, H, N, d, num_sms);
  if (sp.ctas == 0) return classic;
  return {sp.max_pieces, sp.unit0, 2, std::max(classic.workspace, stream_workspace_bytes(sp.ctas, d))};
}

// The 16-bit forward kernel for the head dimension p.d.
cudaError_t launch_fwd16(const fa::FwdParams& p, bool bf16, cudaStream_t s) {
  return p.d == 256 ? fa::launch_fwd_d256(p, bf16, s) : fa::launch_fwd_f16(p, bf16, s);
}

// Argument checks of the forward entry points, in the order their status
// codes are documented: pointers, dtype, shape, head dimension, scale, mask
// flag, size limits, alignment. Nothing here touches a device.
int validate_fwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, int B, int H, int N,
                 int d, float scale, int dtype, int causal) {
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_NULL;
  if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128 && !(d == 256 && dtype != FA_F32)) return FA_ERR_HEADDIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  if (causal != 0 && causal != 1) return FA_ERR_SHAPE;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffLL || BH * N > (1ll << 40) / d) return FA_ERR_SHAPE;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
      (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
    return FA_ERR_ALIGN;
  return FA_OK;
}

int fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
             float scale, int dtype, void* stream, int inject, float* stats_trace, unsigned long long* timeline,
             long long wait_limit, int num_splits = 1, void* workspace = nullptr,
             unsigned long long workspace_bytes = 0, int causal = 0, const int* klen = nullptr,
             float rescale_tau = fa::kRescaleThresholdLog2, float* o_f32 = nullptr) {
  // o_f32 (testing build only): O is written as normalised fp32, before the
  // rounding to the input type, to o_f32 instead of O (O may then be NULL).
  const int vst = validate_fwd(Q, K, V, O ? O : o_f32, LSE, B, H, N, d, scale, dtype, causal);
  if (vst != FA_OK) return vst;
  const long long BH = static_cast<long long>(B) * H;
  if (o_f32 && !aligned16(o_f32)) return FA_ERR_ALIGN;
  if (o_f32 && (dtype == FA_F32 || num_splits != 1 || causal || klen)) return FA_ERR_UNSUPPORTED;
  if (!(rescale_tau >= 0.f) || !(rescale_tau <= 64.f)) return FA_ERR_SCALE;

  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != FA_OK) return st;

  fa::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = Q;
  p.k = K;
  p.v = V;
  p.o = O;
  p.lse = LSE;
  p.status = dev.status;
  p.wait_limit = wait_limit > 0 ? wait_limit : wait_limit_cycles();
  p.inject = inject;
  p.stats_trace = stats_trace;
  p.timeline = timeline;
  p.causal = causal;
  p.klen = klen;
  p.B = B;
  p.H = H;
  p.N = N;
  p.Nk = N;
  p.d = d;
  p.scale = scale;
  p.num_sms = dev.num_sms;
  p.rescale_tau = rescale_tau;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The automatic count of an unmasked 16-bit call may stream the persistent
  // kernel's last units instead of splitting key ranges.
  if (dtype != FA_F32 && num_splits == 0 && !causal && !klen && !o_f32 && inject == 0 && !stats_trace && !timeline) {
    const StreamPlan sp = stream_plan(B, H, N, d, dev.num_sms);
    if (sp.ctas > 0) {
      const unsigned long long need_all = summarize_plan(B, H, N, d, 0, dev.num_sms).workspace;
      if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need_all)
        return FA_ERR_WORKSPACE;
      const unsigned long long rows = 2ull * sp.ctas * kStreamRows;
      p.num_splits = 1;
      p.split_tiles = static_cast<int>(kv_tiles(N, d));
      p.st_unit0 = sp.unit0;
      p.st_tiles = sp.tiles;
      p.st_ctas = sp.ctas;
      p.o_part = static_cast<float*>(workspace);
      p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((rows * d * 4 + 255) & ~255ull));
      FA_DRY_RUN_RETURN();
      const CUtensorMapDataType dt =
          dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
      const int bh = static_cast<int>(BH);
      if (!encode_bhnd_16bit(&p.tm_q, Q, bh, N, d, dt, fa::kF16BlockQ) ||
          !encode_bhnd_16bit(&p.tm_k, K, bh, N, d, dt, fa::kF16BlockKV) ||
          !encode_bhnd_16bit(&p.tm_v, V, bh, N, d, dt, fa::kF16BlockKV) ||
          !encode_bhnd_16bit(&p.tm_o, O, bh, N, d, dt, fa::kF16BlockQ))
        return FA_ERR_CUDA;
      if (!fa::fwd_persist_eligible(p)) return FA_ERR_CUDA;
      const cudaError_t e = fa::launch_fwd_f16(p, dtype == FA_BF16, s);
      return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
  }
  // fp32 always runs unsplit.
  const SplitPlan plan = dtype == FA_F32 ? SplitPlan{1, -1} : split_plan(B, H, N, d, num_splits, dev.num_sms);
  const int splits = plan.splits;
  const long long tiles = kv_tiles(N, d);
  p.split_tiles = static_cast<int>((tiles + splits - 1) / splits);
  p.num_splits = static_cast<int>((tiles + p.split_tiles - 1) / p.split_tiles);
  const long long row0 = (p.num_splits > 1) ? plan_row0(plan, N, d) : 0;
  if (p.num_splits > 1) {
    const unsigned long long need = workspace_bytes_for(B, H, N, d, p.num_splits, row0);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
      return FA_ERR_WORKSPACE;
    const unsigned long long rows = (static_cast<unsigned long long>(B) * H * N - row0) * p.num_splits;
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((rows * d * 4 + 255) & ~255ull));
  }
  if (o_f32) {
    // The one-part epilogue writes [B*H*N, d] fp32 rows and the LSE (natural log).
    p.partial = 1;
    p.o_part = o_f32;
    p.lse_part = LSE;
  }

  FA_DRY_RUN_RETURN();
  cudaError_t e;
  if (dtype == FA_F32) {
    e = fa::launch_fwd_f32(p, s);
  } else {
    const CUtensorMapDataType dt =
        dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int bh = static_cast<int>(BH);
    const int kv_rows = fa::fwd_kv_box_rows(d);
    if (!encode_bhnd_16bit(&p.tm_q, Q, bh, N, d, dt, fa::kF16BlockQ) ||
        !encode_bhnd_16bit(&p.tm_k, K, bh, N, d, dt, kv_rows) ||
        !encode_bhnd_16bit(&p.tm_v, V, bh, N, d, dt, kv_rows) ||
        (O && !encode_bhnd_16bit(&p.tm_o, O, bh, N, d, dt, fa::kF16BlockQ)))
      return FA_ERR_CUDA;
    const bool bf16 = dtype == FA_BF16;
    if (p.num_splits > 1 && plan.tail_qunit0 > 0) {
      // Full waves unsplit (O written directly), then the last wave's units
      // split, then the merge of their rows only.
      const long long qunits = static_cast<long long>(BH) * q_blocks(N, d);
      fa::FwdParams pm = p;
      pm.num_splits = 1;
      pm.split_tiles = static_cast<int>(tiles);
      pm.qunit0 = 0;
      pm.qunit_count = static_cast<int>(plan.tail_qunit0);
      e = launch_fwd16(pm, bf16, s);
      if (e == cudaSuccess) {
        fa::FwdParams pt = p;
        pt.qunit0 = static_cast<int>(plan.tail_qunit0);
        pt.qunit_count = static_cast<int>(qunits - plan.tail_qunit0);
        pt.merge_row0 = row0;
        // The tail's CTAs start as the full waves' CTAs finish instead of at
        // the end of the first launch (they read none of its results).
        pt.launch_pdl = 1;
        e = launch_fwd16(pt, bf16, s);
        if (e == cudaSuccess) e = fa::launch_merge(pt, bf16, s);
      }
    } else {
      e = launch_fwd16(p, bf16, s);
      if (e == cudaSuccess && p.num_splits > 1) e = fa::launch_merge(p, bf16, s);
    }
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// All Nq queries against Nk keys, written as one part of a merge: normalised
// fp32 O and LSE (the split-KV epilogue of the 16-bit kernel, with K and V of
// their own length).
int partial_impl(const void* Q, const void* K, const void* V, float* O_part, float* LSE_part, int B, int H, int Nq,
                 int Nk, int d, float scale, int dtype, void* stream) {
  if (!Q || !K || !V || !O_part || !LSE_part) return FA_ERR_NULL;
  if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (dtype == FA_F32) return FA_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffLL || BH * std::max(Nq, Nk) > (1ll << 40) / d) return FA_ERR_SHAPE;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O_part) ||
      (reinterpret_cast<uintptr_t>(LSE_part) & 3u) != 0)
    return FA_ERR_ALIGN;
  DeviceInfo dev;
  const int st = device_info(&dev);
  if (st != FA_OK) return st;

  fa::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = Q;
  p.k = K;
  p.v = V;
  p.o_part = O_part;
  p.lse_part = LSE_part;
  p.status = dev.status;
  p.wait_limit = wait_limit_cycles();
  p.B = B;
  p.H = H;
  p.N = Nq;
  p.Nk = Nk;
  p.d = d;
  p.scale = scale;
  p.num_sms = dev.num_sms;
  p.rescale_tau = fa::kRescaleThresholdLog2;
  p.num_splits = 1;
  p.split_tiles = static_cast<int>(kv_tiles(Nk, d));
  p.partial = 1;
  const CUtensorMapDataType dt = dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int bh = static_cast<int>(BH);
  if (!encode_bhnd_16bit(&p.tm_q, Q, bh, Nq, d, dt, fa::kF16BlockQ) ||
      !encode_bhnd_16bit(&p.tm_k, K, bh, Nk, d, dt, fa::fwd_kv_box_rows(d)) ||
      !encode_bhnd_16bit(&p.tm_v, V, bh, Nk, d, dt, fa::fwd_kv_box_rows(d)))
    return FA_ERR_CUDA;
  FA_DRY_RUN_RETURN();
  const cudaError_t e = launch_fwd16(p, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int merge_impl(const float* O_parts, const float* LSE_parts, int num_parts, void* O, float* LSE, int B, int H, int N,
               int d, int dtype, void* stream) {
  if (!O_parts || !LSE_parts || !O || !LSE) return FA_ERR_NULL;
  if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (dtype == FA_F32) return FA_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || N < 1 || num_parts < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows * num_parts > (1ll << 40) / d) return FA_ERR_SHAPE;
  if (!aligned16(O_parts) || !aligned16(O) || (reinterpret_cast<uintptr_t>(LSE_parts) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
    return FA_ERR_ALIGN;
  DeviceInfo dev;
  const int st = device_info(&dev);
  if (st != FA_OK) return st;
  fa::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.o_part = const_cast<float*>(O_parts);
  p.lse_part = const_cast<float*>(LSE_parts);
  p.num_splits = num_parts;
  p.o = O;
  p.lse = LSE;
  p.B = B;
  p.H = H;
  p.N = N;
  p.Nk = N;
  p.d = d;
  FA_DRY_RUN_RETURN();
  const cudaError_t e = fa::launch_merge(p, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_fwd_partial(const void* Q, const void* K, const void* V, float* O_part, float* LSE_part, int B, int H, int Nq,
                   int Nk, int d, float scale, int dtype, void* stream) {
  return partial_impl(Q, K, V, O_part, LSE_part, B, H, Nq, Nk, d, scale, dtype, stream);
}

int fa_merge(const float* O_parts, const float* LSE_parts, int num_parts, void* O, float* LSE, int B, int H, int N,
             int d, int dtype, void* stream) {
  return merge_impl(O_parts, LSE_parts, num_parts, O, LSE, B, H, N, d, dtype, stream);
}

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d, float scale,
           int dtype, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream, 0, nullptr, nullptr, 0);
}

int fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
              float scale, int dtype, int causal, const int* seqlens_k, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream, 0, nullptr, nullptr, 0, 1, nullptr, 0, causal,
                  seqlens_k);
}

int fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                   float scale, int dtype, int num_splits, void* workspace, unsigned long long workspace_bytes,
                   void* stream) {
  if (num_splits < 0) return FA_ERR_SHAPE;
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream, 0, nullptr, nullptr, 0, num_splits, workspace,
                  workspace_bytes);
}

int fa_fwd_splitkv_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                      float scale, int dtype, int causal, const int* seqlens_k, int num_splits, void* workspace,
                      unsigned long long workspace_bytes, void* stream) {
  if (num_splits < 0) return FA_ERR_SHAPE;
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream, 0, nullptr, nullptr, 0, num_splits, workspace,
                  workspace_bytes, causal, seqlens_k);
}

int fa_fwd_splitkv_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                           int d, float scale, int dtype, int num_splits, void* stream) {
  // Every argument check of fa_fwd_splitkv first (same codes, same order);
  // only then the device lookup of the scratch and the size limit.
  const int vst = validate_fwd(Q, K, V, O, LSE, B, H, N, d, scale, dtype, 0);
  if (vst != FA_OK) return vst;
  if (num_splits < 0) return FA_ERR_SHAPE;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != FA_OK) return st;
  const unsigned long long need = dtype == FA_F32 ? 0ull : fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits);
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream, 0, nullptr, nullptr, 0, num_splits, scratch,
                  FA_NOALLOC_SCRATCH_BYTES);
}

int fa_fwd_splitkv_launches(int B, int H, int N, int d, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || num_splits < 0) return -FA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return -FA_ERR_HEADDIM;
  DeviceInfo dev;
  const int st = device_info(&dev);
  if (st != FA_OK) return -st;
  return summarize_plan(B, H, N, d, num_splits, dev.num_sms).launches;
}

int fa_fwd_splitkv_plan(int B, int H, int N, int d, int num_splits, int num_sms, int* splits,
                        long long* first_split_unit, int* launches, unsigned long long* workspace_bytes) {
  if (!splits || !first_split_unit || !launches || !workspace_bytes) return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1 || num_splits < 0 || num_sms < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_SHAPE;
  const PlanSummary ps = summarize_plan(B, H, N, d, num_splits, num_sms);
  *splits = ps.splits;
  *first_split_unit = ps.first_split;
  *launches = ps.launches;
  *workspace_bytes = ps.workspace;
  return FA_OK;
}

int fa_fwd_stream_plan(int B, int H, int N, int d, int num_sms, int* unit0, int* tiles, int* ctas) {
  if (!unit0 || !tiles || !ctas) return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1 || num_sms < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_SHAPE;
  const StreamPlan sp = stream_plan(B, H, N, d, num_sms);
  *unit0 = sp.unit0;
  *tiles = sp.tiles;
  *ctas = sp.ctas;
  return FA_OK;
}

int fa_fwd_splitkv_num_splits(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return -FA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return -FA_ERR_HEADDIM;
  DeviceInfo dev;
  const int st = device_info(&dev);
  if (st != FA_OK) return -st;
  return summarize_plan(B, H, N, d, 0, dev.num_sms).splits;
}

unsigned long long fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128 && d != 256) || num_splits < 0) return 0;
  int num_sms = 1;  // an explicit split count does not depend on the device
  if (num_splits == 0) {
    DeviceInfo dev;
    if (device_info(&dev) != FA_OK) return 0;
    num_sms = dev.num_sms;
  }
  return summarize_plan(B, H, N, d, num_splits, num_sms).workspace;
}

}  // extern "C"

namespace {

// fa_bwd workspace: fp32 dQ accumulator [B*H, N, d], then LSE*log2(e) and D
// per row of the 128-row padded layout [B*H, n_pad], each part 256-byte aligned.
unsigned long long bwd_part_bytes(unsigned long long n) { return (n + 255) & ~255ull; }

int bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE, void* dQ,
             void* dK, void* dV, int B, int H, int N, int d, float scale, int dtype, void* workspace,
             unsigned long long workspace_bytes, void* stream, int inject, unsigned long long* timeline,
             long long wait_limit, int causal, const int* seqlens_k) {
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return FA_ERR_NULL;
  if (causal != 0 && causal != 1) return FA_ERR_SHAPE;
  if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (dtype == FA_F32) return FA_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffLL || BH * N > (1ll << 40) / d) return FA_ERR_SHAPE;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV) || (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
    return FA_ERR_ALIGN;
  const unsigned long long need = fa_bwd_workspace_size(B, H, N, d);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return FA_ERR_WORKSPACE;

  DeviceInfo dev;
  const int st = device_info(&dev);
  if (st != FA_OK) return st;

  fa::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.o = O;
  p.dout = dO;
  p.lse = LSE;
  p.dq = dQ;
  p.B = B;
  p.H = H;
  p.N = N;
  p.d = d;
  p.scale = scale;
  p.n_pad = static_cast<int>(bwd_tiles(N) * fa::kF16BlockKV);
  p.status = dev.status;
  p.wait_limit = wait_limit > 0 ? wait_limit : wait_limit_cycles();
  p.inject = inject;
  p.timeline = timeline;
  p.causal = causal;
  p.klen = seqlens_k;
  p.dk = dK;
  p.dv = dV;
  const unsigned long long acc_bytes = bwd_part_bytes(static_cast<unsigned long long>(BH) * N * d * 4);
  const unsigned long long row_bytes = bwd_part_bytes(static_cast<unsigned long long>(BH) * p.n_pad * 4);
  p.dq_acc = static_cast<float*>(workspace);
  p.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes);
  p.dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes + row_bytes);

  const CUtensorMapDataType dt = dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int bh = static_cast<int>(BH);
  // Q tiles of the backward: 128 rows (64 at d = 256); key tiles: 128 rows.
  const int q_rows = d == 256 ? 64 : fa::kF16BlockQ;
  if (!encode_bhnd_16bit(&p.tm_q, Q, bh, N, d, dt, q_rows) ||
      !encode_bhnd_16bit(&p.tm_k, K, bh, N, d, dt, fa::kF16BlockKV) ||
      !encode_bhnd_16bit(&p.tm_v, V, bh, N, d, dt, fa::kF16BlockKV) ||
      !encode_bhnd_16bit(&p.tm_do, dO, bh, N, d, dt, q_rows) ||
      !encode_bhnd_16bit(&p.tm_dk, dK, bh, N, d, dt, fa::kF16BlockKV) ||
      !encode_bhnd_16bit(&p.tm_dv, dV, bh, N, d, dt, fa::kF16BlockKV) ||
      !encode_bhnd_f32_box32(&p.tm_dqacc, p.dq_acc, bh, N, d))
    return FA_ERR_CUDA;
  FA_DRY_RUN_RETURN();
  const cudaError_t e = fa::launch_bwd_f16(p, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

unsigned long long fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128 && d != 256)) return 0;
  const unsigned long long bh = static_cast<unsigned long long>(B) * H;
  const unsigned long long n_pad = static_cast<unsigned long long>(bwd_tiles(N)) * fa::kF16BlockKV;
  return bwd_part_bytes(bh * N * d * 4) + 2 * bwd_part_bytes(bh * n_pad * 4);
}

int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE, void* dQ,
           void* dK, void* dV, int B, int H, int N, int d, float scale, int dtype, void* workspace,
           unsigned long long workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, workspace, workspace_bytes, stream, 0,
                  nullptr, 0, 0, nullptr);
}

int fa_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE, void* dQ,
              void* dK, void* dV, int B, int H, int N, int d, float scale, int dtype, int causal,
              const int* seqlens_k, void* workspace, unsigned long long workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, workspace, workspace_bytes, stream, 0,
                  nullptr, 0, causal, seqlens_k);
}

#ifdef FA_TESTING
int fa_bwd_testing(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                   void* dQ, void* dK, void* dV, int B, int H, int N, int d, float scale, int dtype, void* workspace,
                   unsigned long long workspace_bytes, void* stream, int inject, unsigned long long* timeline,
                   long long wait_limit_cycles) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, workspace, workspace_bytes, stream,
                  inject, timeline, wait_limit_cycles, 0, nullptr);
}
#endif

#ifdef FA_TESTING
int fa_fwd_testing(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                   float scale, int dtype, void* stream, int inject, float* stats_trace,
                   unsigned long long* timeline, long long wait_limit_cycles) {
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream, inject, stats_trace, timeline,
                  wait_limit_cycles);
}

int fa_fwd_debug(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                 float scale, int dtype, void* stream, float* O_f32, float rescale_threshold_log2,
                 float* stats_trace) {
  const float tau = rescale_threshold_log2 < 0.f ? fa::kRescaleThresholdLog2 : rescale_threshold_log2;
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream, 0, stats_trace, nullptr, 0, 1, nullptr, 0, 0,
                  nullptr, tau, O_f32);
}

void fa_testing_set_dry_run(int on) { g_dry_run.store(on ? 1 : 0); }

int fa_testing_stream_piece(int tiles, int ctas, int n, int c, int q, int* out) {
  if (!out || tiles < 1 || ctas < 1 || n < 1 || static_cast<long long>(tiles) * ctas >= (1ll << 31)) return -1;
  if (q < 0) {
    if (c < 0 || static_cast<long long>(c) * n >= tiles) return -1;
    fa::st_unit_ctas(tiles, ctas, n, c, out[0], out[1]);
    return 1;
  }
  if (c < 0 || c >= ctas) return -1;
  fa::StPiece pc;
  if (!fa::st_piece(tiles, ctas, n, c, q, pc)) return 0;
  out[0] = pc.i;
  out[1] = pc.t0;
  out[2] = pc.t1;
  out[3] = pc.slot;
  return 1;
}

int fa_testing_bwd_tile(int B, int H, int N, int d, int causal, int cta, int* out) {
  if (!out || B < 1 || H < 1 || N < 1 || (d != 64 && d != 128 && d != 256)) return -1;
  const long long nt = (static_cast<long long>(N) + 127) / 128;
  const long long ctas = static_cast<long long>(B) * H * nt;
  if (ctas >= (1ll << 31) || cta < 0 || cta >= ctas) return -1;
  const fa::BwdTileOf t = fa::bwd_tile_of(cta, B * H, static_cast<int>(nt), N, d, causal != 0);
  out[0] = t.bh;
  out[1] = t.kt;
  return 1;
}

int fa_testing_fwd_unit(int B, int H, int N, int d, int causal, int num_sms, int unit, int* out) {
  if (!out || B < 1 || H < 1 || N < 1 || num_sms < 0 || (d != 64 && d != 128 && d != 256)) return -1;
  const long long rows = d == 256 ? 128 : 256;
  const long long nqb = (static_cast<long long>(N) + rows - 1) / rows;
  const long long units = static_cast<long long>(B) * H * nqb;
  if (units >= (1ll << 31) || unit < 0 || unit >= units) return -1;
  const fa::FwdUnitOf u = fa::fwd_unit_of(unit, B * H, static_cast<int>(nqb), N, d, causal != 0, num_sms);
  out[0] = u.bh;
  out[1] = u.qb;
  return 1;
}

unsigned int fa_testing_last_timeout_where(void) {
  unsigned int h[2] = {0, 0};
  if (cudaMemcpyFromSymbol(h, g_fa_status, sizeof(h)) != cudaSuccess) return 0xffffffffu;
  return h[1];
}
#endif

int fa_get_device_status(void* stream) {
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int h[2] = {0, 0};
  if (cudaMemcpyFromSymbol(h, g_fa_status, sizeof(h)) != cudaSuccess) return FA_ERR_CUDA;
  if (h[0] == 0) return FA_OK;
  const unsigned int zero[2] = {0, 0};
  if (cudaMemcpyToSymbol(g_fa_status, zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  return (h[0] & fa::kStatusSmemAlign) ? FA_ERR_DEVICE_SMEM : FA_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
