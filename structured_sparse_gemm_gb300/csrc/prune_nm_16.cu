// prune_nm_16.cu -- N:M prune into 2:4 forms for the 16-bit element types,
// and the entry that dispatches on the element type.
#include "prune_nm.cuh"

namespace st24 {

st24_status launch_prune_compress_nm(int dt, int n, int m, bool two, const void* W, int64_t M, int64_t K,
                                     int64_t ldw, void* values, void* meta, cudaStream_t stream) {
  const DeviceInfo* dev = current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  bool ok = false;
  switch (dt) {
    case kF16: ok = prune::launch_nm<kF16, 2>(n, m, two, W, M, K, ldw, values, meta, dev->num_sms, stream); break;
    case kBF16: ok = prune::launch_nm<kBF16, 2>(n, m, two, W, M, K, ldw, values, meta, dev->num_sms, stream); break;
    case kE4M3:
    case kS8: ok = prune::launch_nm_8bit(dt, n, m, two, W, M, K, ldw, values, meta, dev->num_sms, stream); break;
    default: break;
  }
  if (!ok) return ST24_ERR_UNSUPPORTED;
  return cudaGetLastError() == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

}  // namespace st24
