// spmm_mmasp_f16.cu -- instantiation of the warp-level sparse-MMA SpMM for one element type.
#include "spmm_mmasp.cuh"

namespace st24 {
namespace mmasp {
template <>
st24_status launch_dt<kF16>(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                            cudaStream_t s) {
  return launch_dt_impl<kF16>(a, plan, dev, s);
}
}  // namespace mmasp
}  // namespace st24
