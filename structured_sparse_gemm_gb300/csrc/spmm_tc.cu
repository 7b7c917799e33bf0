// spmm_tc.cu -- schedule choice and dispatch of the tcgen05 sparse-MMA SpMM
// (the kernel template lives in spmm_tc.cuh; one translation unit per element
// type instantiates it).
#include "spmm_tc.cuh"

namespace st24 {

// Tile width for a given N: the smallest of 16/32/64 that covers N, else 128.
static int pick_bn_tc(int64_t N) {
  if (N <= 16) return 16;
  if (N <= 32) return 32;
  if (N <= 64) return 64;
  return 128;
}

// N of a CTA-pair tile: 224 (the widest whose two accumulators and the
// metadata ring fit in TMEM), or 128 when that pads N less, weighing 128's
// higher staging cost per output element (34 KB vs 46 KB per stage for
// 128 x 128 vs 128 x 224 outputs per CTA, about 1.29x per element).
static int pick_bnp(int64_t N) {
  const int64_t c224 = (N + 223) / 224 * 224 * 100;
  const int64_t c128 = (N + 127) / 128 * 128 * 129;
  return c128 < c224 ? 128 : 224;
}

StreamKPlan plan_spmm_tc(const SpmmArgs& a, int num_sms) {
  const int bk = elem_size(a.ab) == 2 ? 128 : 256;
  const double a_row = a.K * (elem_size(a.ab) / 2.0 + 0.125), b_col = static_cast<double>(a.K) * elem_size(a.ab);
  const int bn = pick_bn_tc(a.N);
  if (bn < 128) return make_stream_k_plan(128, bn, bk, a.M, a.N, a.K, num_sms, a_row, b_col, false);
  // Wide N: M = 256 tiles on CTA pairs, scheduled over num_sms / 2 pairs.
  // Each CTA keeps its own partial tile and counter, so a pair needs two
  // counters per tile.
  StreamKPlan pl = make_stream_k_plan(256, pick_bnp(a.N), bk, a.M, a.N, a.K, num_sms / 2, a_row, b_col, false);
  pl.pair = 1;
  if (pl.ws_bytes > 0)
    pl.ws_bytes = 2 * static_cast<size_t>(pl.grid) * pl.partial_bytes +
                  (static_cast<size_t>(pl.tiles_m * pl.tiles_n) * 2 * 4 + 255) / 256 * 256;
  return pl;
}

st24_status launch_spmm_tc(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                           cudaStream_t stream) {
  switch (a.ab) {
    case kF16: return tc::launch_dt<kF16>(a, plan, dev, stream);
    case kBF16: return tc::launch_dt<kBF16>(a, plan, dev, stream);
    case kE4M3: return tc::launch_dt<kE4M3>(a, plan, dev, stream);
    default: return ST24_ERR_UNSUPPORTED;
  }
}

}  // namespace st24
