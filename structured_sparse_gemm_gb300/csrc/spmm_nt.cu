// spmm_nt.cu -- schedule and dispatch of the narrow-N tcgen05 SpMM (the kernel
// template lives in spmm_nt.cuh; one translation unit per element type
// instantiates it).
#include "spmm_nt_launch.cuh"

namespace st24 {

namespace {
// The MMA's N for a product of N columns: the smallest multiple of 16 that covers it.
int pick_bn_nt(int64_t N) { return N <= 16 ? 16 : (N <= 32 ? 32 : (N <= 48 ? 48 : 64)); }
}  // namespace

// 8-bit values come in 128-byte chunks of 256 K: K must fill whole chunks.
bool narrow_applies(const SpmmArgs& a) {
  return (a.ab == kF16 || a.ab == kBF16 || (a.ab == kE4M3 && a.K % 256 == 0)) && a.N >= 1 && a.N <= 64;
}

// Each 128-row tile's K range split evenly over a cluster of S CTAs: the
// largest S (a power of two, at most 8 and at most the tile's k-blocks) that
// keeps the grid within ~1.7 CTAs per SM (measured on GB300: 4096-row
// weights run best on 8 CTAs per tile, 11008-row ones on 2, 28672-row ones
// unsplit).  No workspace.
StreamKPlan plan_spmm_nt(const SpmmArgs& a, int num_sms) {
  StreamKPlan pl{};
  pl.bm = 128;
  pl.bn = pick_bn_nt(a.N);
  pl.tiles_m = (a.M + 127) / 128;
  pl.tiles_n = 1;
  // The split S is chosen on the finer stages of split tiles, then the
  // k-block is the stage of the configuration S selects.
  const int64_t fine_iters = (a.K + nt::stage_k(elem_size(a.ab), pl.bn, true) - 1) / nt::stage_k(elem_size(a.ab), pl.bn, true);
  int S = 1;
  while (S < 8 && 2 * S <= fine_iters && pl.tiles_m * 2 * S * 10 <= 17 * static_cast<int64_t>(num_sms)) S *= 2;
  pl.bk = nt::stage_k(elem_size(a.ab), pl.bn, S > 1);
  pl.k_iters = (a.K + pl.bk - 1) / pl.bk;
  pl.cluster = S;
  pl.grid = static_cast<int>(pl.tiles_m * S);
  pl.dp_tiles = pl.tiles_m;
  pl.sk_tiles = 0;
  pl.group_m = 1;
  pl.pair = 0;
  pl.partial_bytes = 0;
  pl.ws_bytes = 0;
  return pl;
}

st24_status launch_spmm_nt(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                           cudaStream_t stream) {
  switch (a.ab) {
    case kF16: return nt::launch_dt<kF16>(a, plan, dev, stream);
    case kBF16: return nt::launch_dt<kBF16>(a, plan, dev, stream);
    case kE4M3: return nt::launch_dt<kE4M3>(a, plan, dev, stream);
    default: return ST24_ERR_UNSUPPORTED;
  }
}

}  // namespace st24
