// spmm_nt_bf16.cu -- instantiation of the narrow-N tcgen05 SpMM for one element type.
#include "spmm_nt_launch.cuh"

namespace st24 {
namespace nt {
template <>
st24_status launch_dt<kBF16>(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev, cudaStream_t s) {
  return launch_dt_impl<kBF16>(a, plan, dev, s);
}
}  // namespace nt
}  // namespace st24
