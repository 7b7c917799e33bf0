// spmm_t_f16.cu -- instantiation of the transposed-use kernel for one element type.
#include "spmm_t_launch.cuh"

namespace st24 {
namespace spt {
template <>
st24_status launch_dt<kF16>(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  return launch_dt_impl<kF16>(a, dev, s);
}
}  // namespace spt
}  // namespace st24
