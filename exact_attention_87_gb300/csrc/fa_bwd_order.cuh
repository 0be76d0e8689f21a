// The order in which the backward pass's main kernels take their key tiles:
// CTA number -> (b*h, key tile). Shared by the d = 64/128 kernel, the two
// d = 256 kernels and the testing build's host-side check.
//
// No causal mask: consecutive CTAs take consecutive key tiles of one head,
// so that all of them read that head's Q, dO and row statistics from L2
// while they run side by side.
//
// Causal mask: key tile t visits the nt - t Q tiles from its diagonal on, so
// CTA lengths run from nt tiles down to one. Taking a head's key tiles in a
// row puts a head's long and short CTAs next to one another; instead the
// CTAs are dealt out longest first within windows of heads (key tile 0 of
// every head of the window, then key tile 1, ...), and each window's heads
// hold at most kBwdWindowBytes of Q, dO and fp32 dQ accumulator (8 N d
// bytes per head: 16 heads at N = 4096, d = 128), so that a window's data
// stays in L2 (129 MB) while its CTAs run. The last window may hold fewer
// heads. Measured on B=8 H=32 N=4096 (causal backward): 886 -> 1016 TFLOP/s
// at d = 128 with 16 heads a window (4: 898, 64: 966-982, all 256: 659),
// 517 -> 610 at d = 64 (32 heads).
#ifndef FA_BWD_ORDER_CUH_
#define FA_BWD_ORDER_CUH_

namespace fa {

constexpr long long kBwdWindowBytes = 64ll << 20;

struct BwdTileOf {
  int bh, kt;
};

// cta in [0, bhn * nt), bhn * nt < 2^31 (the launch checks it); d is the head dimension.
__host__ __device__ inline BwdTileOf bwd_tile_of(int cta, int bhn, int nt, int N, int d, bool causal) {
  BwdTileOf r;
  if (!causal) {
    r.bh = cta / nt;
    r.kt = cta - r.bh * nt;
    return r;
  }
  // 32-bit division only (a 64-bit one is a long routine on the device)
  const long long per_head = 8ll * N * d;
  int win = per_head >= kBwdWindowBytes
                ? 1
                : static_cast<int>(static_cast<unsigned>(kBwdWindowBytes) / static_cast<unsigned>(per_head));
  if (win > bhn) win = bhn;
  const int h0 = cta / (win * nt) * win;        // first head of this CTA's window
  const int g = bhn - h0 < win ? bhn - h0 : win;  // heads in the window
  const int c = cta - h0 * nt;                    // position within the window
  r.kt = c / g;
  r.bh = h0 + (c - r.kt * g);
  return r;
}

}  // namespace fa

#endif  // FA_BWD_ORDER_CUH_
