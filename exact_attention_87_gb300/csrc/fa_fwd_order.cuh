// The order in which the one-CTA-per-unit forward kernels (d = 64/128 and
// d = 256) take their work units (b*h, Q block): unit number -> (b*h, Q
// block). Shared by both kernels and the testing build's host-side check.
//
// Unmasked, and every split or partial launch: a head's Q blocks come in a
// row (unit = bh * nqb + qb), so the CTAs running side by side share that
// head's K and V in L2, and the split-KV tail plan's units (the last ones)
// hold the last rows.
//
// Causal, one launch over every unit unsplit: Q block qb sees (qb + 1)
// blocks' worth of keys, so units run from one tile to nqb. They are dealt
// out longest first within windows of heads (the last Q block of every head
// of the window, then the one before, ...), each window's heads holding at
// most kFwdWindowBytes of K and V (4 Nk d bytes per head: 32 heads at
// Nk = 4096, d = 128), so that a window's K and V stay in L2 (129 MB) while
// its CTAs run; the last window may hold fewer heads. Measured (causal, one
// CTA per unit, same-box A/B against longest first within each head): B=1
// H=8 N=16384 d=128 1282-1293 -> 1527-1555 TFLOP/s; B=8 H=32 N=4096 d=64
// 784 -> 800. A launch whose units all fit on the SMs at once (num_sms > 0
// and units <= num_sms) keeps longest first within each head: on B=1 H=4
// N=512 d=64 causal the windows cost 0.7-1.5 us of an 11 us call (with
// this rule and the 32-bit division below: 10.7-10.9 us, as before them).
#ifndef FA_FWD_ORDER_CUH_
#define FA_FWD_ORDER_CUH_

namespace fa {

constexpr long long kFwdWindowBytes = 64ll << 20;

struct FwdUnitOf {
  int bh, qb;
};

// unit in [0, bhn * nqb) < 2^31; nk = keys per head, d = head dimension,
// num_sms = the device's SM count (0: unknown).
__host__ __device__ inline FwdUnitOf fwd_unit_of(int unit, int bhn, int nqb, int nk, int d, bool causal_whole,
                                                 int num_sms) {
  FwdUnitOf r;
  if (!causal_whole || (num_sms > 0 && bhn * nqb <= num_sms)) {
    r.bh = unit / nqb;
    r.qb = unit - r.bh * nqb;
    if (causal_whole) r.qb = nqb - 1 - r.qb;  // one wave: longest first within each head
    return r;
  }
  // 32-bit division only (a 64-bit one is a long routine on the device)
  const long long per_head = 4ll * (nk > 0 ? nk : 1) * d;
  int win = per_head >= kFwdWindowBytes
                ? 1
                : static_cast<int>(static_cast<unsigned>(kFwdWindowBytes) / static_cast<unsigned>(per_head));
  if (win > bhn) win = bhn;
  const int h0 = unit / (win * nqb) * win;        // first head of this unit's window
  const int g = bhn - h0 < win ? bhn - h0 : win;  // heads in the window
  const int c = unit - h0 * nqb;                  // position within the window
  const int j = c / g;                            // 0: the last (longest) Q block
  r.bh = h0 + (c - j * g);
  r.qb = nqb - 1 - j;
  return r;
}

}  // namespace fa

#endif  // FA_FWD_ORDER_CUH_
