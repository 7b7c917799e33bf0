// spmm_tc_f16.cu -- instantiation of the tcgen05 sparse-MMA SpMM for one element type.
#include "spmm_tc.cuh"

namespace st24 {
namespace tc {
template <>
st24_status launch_dt<kF16>(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                          cudaStream_t s) {
  return launch_dt_impl<kF16>(a, plan, dev, s);
}
}  // namespace tc
}  // namespace st24
