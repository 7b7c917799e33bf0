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
static int pick_bnp(int64_t N, int elem_bytes) {
  // e4m3 at N = 449..512: two 256-column tiles (one accumulator, 3 stages)
  // instead of four 128-column ones: 74.8 -> 70.9 us on 28672x8192 at
  // N = 512, 29.2 -> 26.7 us on 8192x8192 (bf16 measured slower).
  if (elem_bytes == 1 && N > 448 && N <= 512) return 256;
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
  // Costs in k-blocks of MMA time per pair.  Whole tiles in data-parallel
  // waves cost waves * k_iters.  Splitting a tile s ways over K costs
  // k_iters / s plus finishing it: the partials go through the workspace and
  // the last contributor sums them, about 50 + 23 s k-blocks (measured).  So
  // tiles are split only when they are fewer than the pairs and long: a
  // stream-K tail after full waves never pays (11008x4096 at N = 600, 1000
  // and 2048 and 4096x4096 at N = 2048 ran 1.7-2.6x faster as data-parallel
  // waves), nor does a split over all the pairs (256x32768 at N = 200 took 8x
  // the unsplit time split 76 ways).
  const int pairs = num_sms / 2;
  const int bnp = pick_bnp(a.N, elem_size(a.ab));
  const int64_t tiles = ((a.M + 255) / 256) * ((a.N + bnp - 1) / bnp);
  const int64_t KI = (a.K + bk - 1) / bk;
  double best = static_cast<double>((tiles + pairs - 1) / (pairs > 0 ? pairs : 1)) * static_cast<double>(KI);
  int64_t best_s = 1;
  for (int64_t sp = 2; tiles > 0 && sp * tiles <= pairs; ++sp) {
    const double cost = static_cast<double>(KI) / sp + 50.0 + 23.0 * sp;
    if (cost < best) { best = cost; best_s = sp; }
  }
  // A grid of tiles * best_s pairs: every tile split best_s ways (whole
  // tiles when best_s is 1), each pair taking one contiguous run of k-blocks.
  const int64_t g = best_s > 1 ? tiles * best_s : (tiles < pairs ? (tiles > 0 ? tiles : 1) : pairs);
  StreamKPlan pl = make_stream_k_plan(256, bnp, bk, a.M, a.N, a.K, static_cast<int>(g), a_row, b_col, false);
  pl.pair = 1;
  if (best_s == 1 && tiles > pl.grid) {   // full waves: never a stream-K tail
    pl.dp_tiles = tiles;
    pl.sk_tiles = 0;
    pl.ws_bytes = 0;
  }
  // Each CTA keeps its own partial tile and counter, so a pair needs two
  // counters per tile.
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
