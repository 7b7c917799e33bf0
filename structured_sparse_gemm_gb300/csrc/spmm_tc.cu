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

StreamKPlan plan_spmm_tc(const SpmmArgs& a, int num_sms) {
  return make_stream_k_plan(128, pick_bn_tc(a.N), elem_size(a.ab) == 2 ? 128 : 256, a.M, a.N, a.K, num_sms,
                            a.K * (elem_size(a.ab) / 2.0 + 0.125), static_cast<double>(a.K) * elem_size(a.ab),
                            false);
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
