// spmm_tc_e4m3.cu -- instantiation of the tcgen05 sparse-MMA SpMM for one element type.
#include "spmm_tc.cuh"

namespace st24 {
namespace tc {
template <>
st24_status launch_dt<kE4M3>(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                          cudaStream_t s) {
  return launch_dt_impl<kE4M3>(a, plan, dev, s);
}
}  // namespace tc
}  // namespace st24
